// attn_noalloc.cu -- a decode entry point that allocates nothing.
//
// Some callers cannot allocate device memory at call time: a serving engine
// that reserves all of HBM for its own pools up front leaves nothing for
// cudaMalloc/cudaMallocAsync to hand out, and a host framework with its own
// caching allocator may forbid other allocators outright; others cannot
// accept the implicit device synchronisation a cudaMalloc/cudaFree may
// cause. attn_fwd_decode_noalloc serves them: it runs the same split-KV decode
// kernels as attn_fwd, but keeps the per-partition partials in a fixed
// array of device memory that belongs to the library (defined below), so the
// caller passes only inputs and outputs.
//
// The array costs ATTN_NOALLOC_SCRATCH_BYTES of memory on every device that
// loads the library, for as long as the library stays loaded. All calls on a
// device share it: two calls whose kernels overlap on the GPU (for example on
// two streams) race on it and produce wrong results. Nothing in it needs to
// start at zero: each call writes every partial it later reads.
#include <cuda_runtime.h>

#include <cstdint>

#include "attn.h"
#include "attn_internal.h"

namespace {

constexpr size_t kScratchFloats = ATTN_NOALLOC_SCRATCH_BYTES / sizeof(float);

// The library's own decode scratch: [B*h][S][d+4] fp32 partials.
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

// Device address of g_decode_scratch on the current device. In host code the
// symbol names a host-side stand-in, not device memory, so the kernels must
// receive this address instead. It is looked up on every call (the lookup
// enqueues nothing): an address kept from an earlier call would go stale if
// the caller reset the device, which reloads the module elsewhere.
float* scratch_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
  return static_cast<float*>(p);
}

}  // namespace

extern "C" attn_status_t attn_fwd_decode_noalloc(const void* q, const void* k, const void* v,
                                                 void* o, float* lse, int B, int h, int T_kv,
                                                 int d, float scale, int dtype, int num_splits,
                                                 void* stream) {
  bool empty = false;
  attn_status_t st = attn::detail::validate(q, k, v, o, lse, B, h, 1, T_kv, d, scale, 0, dtype,
                                            &empty);
  if (st != ATTN_OK) return st;
  if (num_splits < 0 || num_splits > 1024) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  const int bf16 = dtype == ATTN_BF16 ? 1 : 0;
  const int splits =
      num_splits > 0 ? num_splits : attn::detail::choose_splits(static_cast<long long>(B) * h, T_kv, d, 1);
  if (static_cast<long long>(B) * h * splits > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  const size_t need = static_cast<size_t>(B) * h * splits * attn::decode_partial_floats(d);
  if (need > kScratchFloats) return ATTN_ERR_WORKSPACE;  // beyond the fixed scratch
  float* ws = scratch_ptr();
  if (!ws) return ATTN_ERR_CUDA;
  attn::FwdProblem p{q, k, v, o, lse, B, h, 1, T_kv, d, scale, 0, bf16, nullptr, h};
  const char* name = nullptr;
  return attn::launch_decode(p, splits, ws, static_cast<cudaStream_t>(stream), &name) ==
                 cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}
