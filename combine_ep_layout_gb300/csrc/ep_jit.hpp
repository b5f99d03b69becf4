// ep_jit.hpp -- run-time specialisation of the data kernels for shapes that
// have no compiled variant ("MORI JIT v2" §1-§3.4 and the JIT flow of "DeepEP
// overall architecture analysis": configuration -> rendered source -> hash key
// -> compile -> cache -> load -> launch).
//
// The configuration becomes source text (template arguments of the kernel
// bodies in ep_dispatch_body.cuh / ep_combine_body.cuh); the text, the bodies,
// the compiler version and flags make the SHA-256 cache key; NVRTC compiles
// the text for the device's architecture; the cubin is kept on disk under the
// key (published by an atomic rename, so racing processes agree) and loaded
// once per device with the driver API.  NVRTC and the driver are opened with
// dlopen, so the library loads, and its other entry points work, where neither
// exists.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <string>
#include <vector>

#include "ep_types.cuh"

namespace epg {
namespace jit {

// What to specialise.  The launch configuration follows from it.
struct Request {
  enum Kind { kCopy = 0, kFp8 = 1, kCombine = 2 } kind;
  int row_bytes;   // kCopy: bytes per transported row
  int hidden;      // kFp8, kCombine: channels per row
  int topk;
  bool weighted;   // kCombine
};

// A loaded specialisation.  `function` is a CUfunction (kept opaque here).
struct Kernel {
  void* function = nullptr;
  int block = 0;          // threads per CTA
  std::string name;       // entry name, also the variant name reported to users
};

// True when the request has a specialisation worth compiling (a compile-time
// row geometry exists for it).
bool Worthwhile(const Request& r);

// Entry name of the specialisation, e.g. "ep_jit_dispatch_copy_rb6144_k5".
std::string EntryName(const Request& r);

// Source text of the translation unit for the request.
std::string RenderSource(const Request& r);

// Make the cubin for `r` available in the disk cache (compiling it when
// missing) for architecture `arch` ("sm_103a").  *compiled tells whether this
// call compiled it; *entry_dir receives the cache entry's directory.  Returns
// false with *err on failure (no NVRTC, compile error, file system error).
bool Prepare(const Request& r, const std::string& arch, bool* compiled, std::string* entry_dir,
             std::string* err);

// Prepare for the current device and load the function into its context.
bool Load(const Request& r, Kernel* out, std::string* err);

// Launch a loaded kernel with one argument block (DispatchParams or
// CombineParams) on `stream`.
cudaError_t Launch(const Kernel& k, int grid, const void* params, cudaStream_t stream);

// False when run-time specialisation is switched off (EP_GB300_JIT=0).
bool Enabled();

// SHA-256 of `data`, lower-case hex (FIPS 180-4).
std::string Sha256Hex(const std::string& data);

}  // namespace jit
}  // namespace epg
