// ep_jit.cpp -- run-time specialisation: render, key, compile, cache, load,
// launch (see ep_jit.hpp).
#include "ep_jit.hpp"

#include <cuda.h>
#include <dlfcn.h>
#include <errno.h>
#include <fcntl.h>
#include <nvrtc.h>
#include <sys/stat.h>
#include <unistd.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "ep_cfg.hpp"
#include "ep_kernels.hpp"

namespace epg {
namespace jit {

namespace {

// ------------------------------------------------------------------ SHA-256

// SHA-256 as specified in FIPS 180-4.  The round constants and the initial
// hash value are derived from their definition (the first 32 bits of the
// fractional parts of the cube roots of the first 64 primes, and of the square
// roots of the first 8 primes) with exact integer arithmetic, not typed in.
struct Sha256Consts {
  uint32_t k[64];
  uint32_t h0[8];
  Sha256Consts() {
    int primes[64];
    int n = 0;
    for (int c = 2; n < 64; ++c) {
      bool prime = true;
      for (int d = 2; d * d <= c; ++d)
        if (c % d == 0) { prime = false; break; }
      if (prime) primes[n++] = c;
    }
    using u128 = unsigned __int128;
    for (int i = 0; i < 64; ++i) {  // largest m with m^3 <= p * 2^96: m = floor(cbrt(p) * 2^32)
      const u128 target = static_cast<u128>(primes[i]) << 96;
      uint64_t lo = 0, hi = 1ull << 36;
      while (lo < hi) {
        const uint64_t mid = lo + (hi - lo + 1) / 2;
        if (static_cast<u128>(mid) * mid * mid <= target) lo = mid; else hi = mid - 1;
      }
      k[i] = static_cast<uint32_t>(lo);  // the fractional part's first 32 bits
    }
    for (int i = 0; i < 8; ++i) {  // largest m with m^2 <= p * 2^64
      const u128 target = static_cast<u128>(primes[i]) << 64;
      uint64_t lo = 0, hi = 1ull << 36;
      while (lo < hi) {
        const uint64_t mid = lo + (hi - lo + 1) / 2;
        if (static_cast<u128>(mid) * mid <= target) lo = mid; else hi = mid - 1;
      }
      h0[i] = static_cast<uint32_t>(lo);
    }
  }
};

const Sha256Consts& consts() {
  static const Sha256Consts c;
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void sha256_block(uint32_t h[8], const uint8_t* b) {
  const uint32_t* K = consts().k;
  uint32_t w[64];
  for (int i = 0; i < 16; ++i)
    w[i] = (uint32_t(b[4 * i]) << 24) | (uint32_t(b[4 * i + 1]) << 16) | (uint32_t(b[4 * i + 2]) << 8) |
           uint32_t(b[4 * i + 3]);
  for (int i = 16; i < 64; ++i) {
    const uint32_t s0 = rotr(w[i - 15], 7) ^ rotr(w[i - 15], 18) ^ (w[i - 15] >> 3);
    const uint32_t s1 = rotr(w[i - 2], 17) ^ rotr(w[i - 2], 19) ^ (w[i - 2] >> 10);
    w[i] = w[i - 16] + s0 + w[i - 7] + s1;
  }
  uint32_t a = h[0], bb = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
  for (int i = 0; i < 64; ++i) {
    const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t t1 = hh + S1 + ch + K[i] + w[i];
    const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    const uint32_t maj = (a & bb) ^ (a & c) ^ (bb & c);
    const uint32_t t2 = S0 + maj;
    hh = g; g = f; f = e; e = d + t1; d = c; c = bb; bb = a; a = t1 + t2;
  }
  h[0] += a; h[1] += bb; h[2] += c; h[3] += d; h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
}

// ---------------------------------------------------- dynamic libraries

struct Nvrtc {
  decltype(&nvrtcCreateProgram) create = nullptr;
  decltype(&nvrtcCompileProgram) compile = nullptr;
  decltype(&nvrtcGetProgramLogSize) log_size = nullptr;
  decltype(&nvrtcGetProgramLog) log = nullptr;
  decltype(&nvrtcGetCUBINSize) cubin_size = nullptr;
  decltype(&nvrtcGetCUBIN) cubin = nullptr;
  decltype(&nvrtcDestroyProgram) destroy = nullptr;
  decltype(&nvrtcVersion) version = nullptr;
  bool ok = false;
};

void* open_first(const std::vector<std::string>& names) {
  for (const auto& n : names)
    if (void* h = dlopen(n.c_str(), RTLD_NOW | RTLD_LOCAL)) return h;
  return nullptr;
}

const Nvrtc& nvrtc() {
  static Nvrtc n = [] {
    Nvrtc r;
    std::vector<std::string> names = {"libnvrtc.so.13", "libnvrtc.so"};
    if (const char* home = std::getenv("CUDA_HOME")) names.push_back(std::string(home) + "/lib64/libnvrtc.so.13");
    names.push_back("/usr/local/cuda/lib64/libnvrtc.so.13");
    void* h = open_first(names);
    if (!h) return r;
#define EPG_SYM(field, name) r.field = reinterpret_cast<decltype(r.field)>(dlsym(h, name))
    EPG_SYM(create, "nvrtcCreateProgram");
    EPG_SYM(compile, "nvrtcCompileProgram");
    EPG_SYM(log_size, "nvrtcGetProgramLogSize");
    EPG_SYM(log, "nvrtcGetProgramLog");
    EPG_SYM(cubin_size, "nvrtcGetCUBINSize");
    EPG_SYM(cubin, "nvrtcGetCUBIN");
    EPG_SYM(destroy, "nvrtcDestroyProgram");
    EPG_SYM(version, "nvrtcVersion");
#undef EPG_SYM
    r.ok = r.create && r.compile && r.log_size && r.log && r.cubin_size && r.cubin && r.destroy &&
           r.version;
    return r;
  }();
  return n;
}

struct Driver {
  decltype(&cuModuleLoadData) load = nullptr;
  decltype(&cuModuleGetFunction) get_function = nullptr;
  decltype(&cuLaunchKernel) launch = nullptr;
  decltype(&cuLaunchKernelEx) launch_ex = nullptr;  // for programmatic dependent launch
  bool ok = false;
};

const Driver& driver() {
  static Driver d = [] {
    Driver r;
    void* h = open_first({"libcuda.so.1", "libcuda.so"});
    if (!h) return r;
    r.load = reinterpret_cast<decltype(r.load)>(dlsym(h, "cuModuleLoadData"));
    r.get_function = reinterpret_cast<decltype(r.get_function)>(dlsym(h, "cuModuleGetFunction"));
    r.launch = reinterpret_cast<decltype(r.launch)>(dlsym(h, "cuLaunchKernel"));
    r.launch_ex = reinterpret_cast<decltype(r.launch_ex)>(dlsym(h, "cuLaunchKernelEx"));
    r.ok = r.load && r.get_function && r.launch;
    return r;
  }();
  return d;
}

// ------------------------------------------------------------- sources

// The kernel bodies live beside this library (csrc/ next to libep_gb300.so),
// so the text that is compiled is the text this library was built from.
void anchor() {}

std::string source_dir() {
  Dl_info info;
  if (dladdr(reinterpret_cast<void*>(&anchor), &info) && info.dli_fname) {
    std::string lib = info.dli_fname;
    const size_t slash = lib.rfind('/');
    return (slash == std::string::npos ? std::string(".") : lib.substr(0, slash)) + "/csrc";
  }
  return "csrc";
}

bool read_file(const std::string& path, std::string* out) {
  FILE* f = std::fopen(path.c_str(), "rb");
  if (!f) return false;
  std::string s;
  char buf[1 << 16];
  size_t n;
  while ((n = std::fread(buf, 1, sizeof buf, f)) > 0) s.append(buf, n);
  std::fclose(f);
  *out = std::move(s);
  return true;
}

const char* const kHeaders[] = {"ep_cfg.hpp", "ep_types.cuh", "ep_dispatch_body.cuh",
                                "ep_combine_body.cuh"};
constexpr int kNumHeaders = 4;

struct HeaderSet {
  std::string text[kNumHeaders];
  std::string digest;
  bool ok = false;
  std::string err;
};

const HeaderSet& headers() {
  static HeaderSet hs = [] {
    HeaderSet r;
    const std::string dir = source_dir();
    std::string all;
    for (int i = 0; i < kNumHeaders; ++i) {
      if (!read_file(dir + "/" + kHeaders[i], &r.text[i])) {
        r.err = "cannot read kernel source " + dir + "/" + kHeaders[i];
        return r;
      }
      all += kHeaders[i];
      all.push_back('\0');
      all += r.text[i];
      all.push_back('\0');
    }
    r.digest = Sha256Hex(all);
    r.ok = true;
    return r;
  }();
  return hs;
}

// Minimum resident CTAs per SM stated in the rendered launch bounds (the copy
// kernel's, as for the compiled variants; 1 elsewhere).
int min_blocks_of(const Request& r) {
  return r.kind == Request::kCopy ? CopyMinBlocks(r.row_bytes, 8) : 1;
}

int block_of(const Request& r) {
  switch (r.kind) {
    case Request::kCopy: return RowThreads(r.row_bytes / 32);
    case Request::kFp8: return RowThreads(2 * r.hidden / 32);
    default: return 128;  // kCombineThreads
  }
}

// ---------------------------------------------------------------- cache

bool mkdirs(const std::string& path) {
  size_t pos = 0;
  while (true) {
    pos = path.find('/', pos + 1);
    const std::string part = path.substr(0, pos);
    if (!part.empty() && mkdir(part.c_str(), 0755) != 0 && errno != EEXIST) return false;
    if (pos == std::string::npos) return true;
  }
}

bool write_file_synced(const std::string& path, const std::string& data) {
  const int fd = open(path.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
  if (fd < 0) return false;
  size_t off = 0;
  while (off < data.size()) {
    const ssize_t w = write(fd, data.data() + off, data.size() - off);
    if (w <= 0) { close(fd); return false; }
    off += static_cast<size_t>(w);
  }
  const bool ok = fsync(fd) == 0;
  return close(fd) == 0 && ok;
}

void remove_dir(const std::string& dir) {
  for (const char* f : {"kernel.cu", "kernel.cubin", "signature.txt"}) unlink((dir + "/" + f).c_str());
  rmdir(dir.c_str());
}

std::string cache_root() {
  if (const char* c = std::getenv("EP_GB300_JIT_CACHE")) return c;
  const char* home = std::getenv("HOME");
  return std::string(home ? home : "/tmp") + "/.cache/ep_gb300/jit";
}

// -default-device: the shared constexpr arithmetic of ep_cfg.hpp carries no
// execution-space annotation (so that a host-only compiler accepts it).
std::string options_text(const std::string& arch) {
  return "--gpu-architecture=" + arch + " -std=c++17 -default-device";
}

bool compile(const Request& r, const std::string& arch, const std::string& src, std::string* cubin,
             std::string* err) {
  const Nvrtc& nv = nvrtc();
  const HeaderSet& hs = headers();
  const char* contents[kNumHeaders];
  for (int i = 0; i < kNumHeaders; ++i) contents[i] = hs.text[i].c_str();
  nvrtcProgram prog;
  if (nv.create(&prog, src.c_str(), "kernel.cu", kNumHeaders, contents, kHeaders) != NVRTC_SUCCESS) {
    *err = "nvrtcCreateProgram failed";
    return false;
  }
  const std::string a = "--gpu-architecture=" + arch;
  const char* opts[] = {a.c_str(), "-std=c++17", "-default-device"};
  const nvrtcResult res = nv.compile(prog, 3, opts);
  if (res != NVRTC_SUCCESS) {
    size_t n = 0;
    nv.log_size(prog, &n);
    std::string log(n, '\0');
    if (n) nv.log(prog, &log[0]);
    *err = "NVRTC failed to compile " + EntryName(r) + ":\n" + log;
    nv.destroy(&prog);
    return false;
  }
  size_t n = 0;
  nv.cubin_size(prog, &n);
  cubin->assign(n, '\0');
  nv.cubin(prog, &(*cubin)[0]);
  nv.destroy(&prog);
  return true;
}

std::atomic<unsigned> g_tmp_counter{0};

struct Loaded {
  CUfunction function;
};
std::mutex g_mu;
std::map<std::pair<int, std::string>, Loaded> g_loaded;  // (device, entry dir) -> function

}  // namespace

std::string Sha256Hex(const std::string& data) {
  uint32_t h[8];
  std::memcpy(h, consts().h0, sizeof h);
  const uint8_t* p = reinterpret_cast<const uint8_t*>(data.data());
  const size_t n = data.size();
  size_t i = 0;
  for (; i + 64 <= n; i += 64) sha256_block(h, p + i);
  uint8_t tail[128] = {0};
  const size_t rem = n - i;
  std::memcpy(tail, p + i, rem);
  tail[rem] = 0x80;
  const size_t tl = rem + 9 <= 64 ? 64 : 128;
  const uint64_t bits = static_cast<uint64_t>(n) * 8;
  for (int b = 0; b < 8; ++b) tail[tl - 1 - b] = static_cast<uint8_t>(bits >> (8 * b));
  sha256_block(h, tail);
  if (tl == 128) sha256_block(h, tail + 64);
  char out[65];
  for (int j = 0; j < 8; ++j) std::snprintf(out + 8 * j, 9, "%08x", h[j]);
  return std::string(out, 64);
}

bool Enabled() {
  const char* e = std::getenv("EP_GB300_JIT");
  return !(e && std::strcmp(e, "0") == 0);
}

bool Worthwhile(const Request& r) {
  switch (r.kind) {
    case Request::kCopy: return r.row_bytes % 32 == 0 && RowThreads(r.row_bytes / 32) > 0;
    case Request::kFp8: return r.hidden % kScaleGroup == 0 && RowThreads(2 * r.hidden / 32) > 0;
    default: return r.hidden % 16 == 0;
  }
}

std::string EntryName(const Request& r) {
  char buf[96];
  switch (r.kind) {
    case Request::kCopy:
      std::snprintf(buf, sizeof buf, "ep_jit_dispatch_copy_rb%d_k%d", r.row_bytes, r.topk);
      break;
    case Request::kFp8:
      std::snprintf(buf, sizeof buf, "ep_jit_dispatch_fp8_h%d_k%d", r.hidden, r.topk);
      break;
    default:
      std::snprintf(buf, sizeof buf, "ep_jit_combine_%sh%d_k%d", r.weighted ? "w_" : "", r.hidden,
                    r.topk);
  }
  return buf;
}

std::string RenderSource(const Request& r) {
  const std::string name = EntryName(r);
  char buf[512];
  switch (r.kind) {
    case Request::kCopy:
      std::snprintf(buf, sizeof buf,
                    "// ep_gb300 run-time specialisation (generated)\n"
                    "#include \"ep_dispatch_body.cuh\"\n"
                    "extern \"C\" __global__ void __launch_bounds__(%d, %d) %s(epg::DispatchParams p) {\n"
                    "  epg::dispatch_copy_body<%d, %d, 8>(p);\n}\n",
                    block_of(r), min_blocks_of(r), name.c_str(), r.row_bytes, r.topk);
      break;
    case Request::kFp8:
      std::snprintf(buf, sizeof buf,
                    "// ep_gb300 run-time specialisation (generated)\n"
                    "#include \"ep_dispatch_body.cuh\"\n"
                    "extern \"C\" __global__ void __launch_bounds__(%d, 1) %s(epg::DispatchParams p) {\n"
                    "  epg::dispatch_fp8_body<%d, %d, 8>(p);\n}\n",
                    block_of(r), name.c_str(), r.hidden, r.topk);
      break;
    default:
      std::snprintf(buf, sizeof buf,
                    "// ep_gb300 run-time specialisation (generated)\n"
                    "#include \"ep_combine_body.cuh\"\n"
                    "extern \"C\" __global__ void __launch_bounds__(%d) %s(epg::CombineParams p) {\n"
                    "  epg::combine_body<%d, %d, %s, 8, false, false>(p);\n}\n",
                    block_of(r), name.c_str(), r.hidden, r.topk, r.weighted ? "true" : "false");
  }
  return buf;
}

bool Prepare(const Request& r, const std::string& arch, bool* compiled, std::string* entry_dir,
             std::string* err) {
  *compiled = false;
  const Nvrtc& nv = nvrtc();
  if (!nv.ok) {
    *err = "NVRTC (libnvrtc.so.13) is not available";
    return false;
  }
  const HeaderSet& hs = headers();
  if (!hs.ok) {
    *err = hs.err;
    return false;
  }
  int major = 0, minor = 0;
  nv.version(&major, &minor);
  const std::string name = EntryName(r);
  const std::string src = RenderSource(r);
  char ver[32];
  std::snprintf(ver, sizeof ver, "nvrtc-%d.%d", major, minor);
  // the key covers everything that decides the binary: entry, compiler,
  // flags, the included kernel bodies and the rendered text
  const std::string signature = name + "$$" + ver + "$$" + options_text(arch) + "$$" + hs.digest +
                                "$$" + src;
  const std::string key = Sha256Hex(signature);
  const std::string root = cache_root();
  const std::string dir = root + "/" + arch + "/kernel." + name + "." + key.substr(0, 16);
  *entry_dir = dir;
  struct stat st;
  if (stat((dir + "/kernel.cubin").c_str(), &st) == 0) return true;  // published before

  std::string cubin;
  if (!compile(r, arch, src, &cubin, err)) return false;
  if (!mkdirs(root + "/" + arch) || !mkdirs(root + "/tmp")) {
    *err = "cannot create the cache directory " + root;
    return false;
  }
  char tmpname[64];
  std::snprintf(tmpname, sizeof tmpname, "/tmp/%d.%u", static_cast<int>(getpid()),
                g_tmp_counter.fetch_add(1));
  const std::string tmp = root + tmpname;
  if (mkdir(tmp.c_str(), 0755) != 0 || !write_file_synced(tmp + "/kernel.cu", src) ||
      !write_file_synced(tmp + "/kernel.cubin", cubin) ||
      !write_file_synced(tmp + "/signature.txt", signature)) {
    remove_dir(tmp);
    *err = "cannot write the cache entry under " + tmp;
    return false;
  }
  if (rename(tmp.c_str(), dir.c_str()) != 0) {
    const int e = errno;
    remove_dir(tmp);
    if (e != EEXIST && e != ENOTEMPTY) {  // anything but "another process published it first"
      *err = "cannot publish the cache entry " + dir + ": " + std::strerror(e);
      return false;
    }
    return true;
  }
  *compiled = true;
  return true;
}

bool Load(const Request& r, Kernel* out, std::string* err) {
  const Driver& drv = driver();
  if (!drv.ok) {
    *err = "the CUDA driver library is not available";
    return false;
  }
  int dev = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaFree(nullptr);  // make the primary context current
  if (e != cudaSuccess) {
    *err = std::string("no usable device: ") + cudaGetErrorString(e);
    return false;
  }
  char arch[16];
  std::snprintf(arch, sizeof arch, "sm_%d%d%s", major, minor, major >= 9 ? "a" : "");
  bool compiled = false;
  std::string dir;
  if (!Prepare(r, arch, &compiled, &dir, err)) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_loaded.find({dev, dir});
  if (it == g_loaded.end()) {
    std::string cubin;
    if (!read_file(dir + "/kernel.cubin", &cubin)) {
      *err = "cannot read " + dir + "/kernel.cubin";
      return false;
    }
    CUmodule mod;
    CUfunction fn;
    if (drv.load(&mod, cubin.data()) != CUDA_SUCCESS) {
      *err = "cuModuleLoadData failed for " + dir;
      return false;
    }
    if (drv.get_function(&fn, mod, EntryName(r).c_str()) != CUDA_SUCCESS) {
      *err = "cuModuleGetFunction failed for " + EntryName(r);
      return false;
    }
    it = g_loaded.emplace(std::make_pair(dev, dir), Loaded{fn}).first;
  }
  out->function = reinterpret_cast<void*>(it->second.function);
  out->block = block_of(r);
  out->name = EntryName(r);
  return true;
}

cudaError_t Launch(const Kernel& k, int grid, const void* params, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  void* args[1] = {const_cast<void*>(params)};
  const Driver& d = driver();
  CUresult r;
  if (d.launch_ex && epg::PdlEnabled()) {
    // programmatic stream serialisation, as for the compiled variants: the
    // kernel bodies wait for the preceding grid before touching memory
    CUlaunchAttribute attr[1];
    attr[0].id = CU_LAUNCH_ATTRIBUTE_PROGRAMMATIC_STREAM_SERIALIZATION;
    attr[0].value.programmaticStreamSerializationAllowed = 1;
    CUlaunchConfig cfg = {};
    cfg.gridDimX = static_cast<unsigned>(grid);
    cfg.gridDimY = cfg.gridDimZ = 1;
    cfg.blockDimX = static_cast<unsigned>(k.block);
    cfg.blockDimY = cfg.blockDimZ = 1;
    cfg.sharedMemBytes = 0;
    cfg.hStream = reinterpret_cast<CUstream>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    r = d.launch_ex(&cfg, reinterpret_cast<CUfunction>(k.function), args, nullptr);
  } else {
    r = d.launch(reinterpret_cast<CUfunction>(k.function), grid, 1, 1, k.block, 1, 1, 0,
                 reinterpret_cast<CUstream>(stream), args, nullptr);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorLaunchFailure;
}

}  // namespace jit
}  // namespace epg
