// merge_sm103.cuh -- the exact merge of key-partition partials of one query
// row, shared by the decode merge kernel and the split-KV prefill kernel's
// fused merge.
//
// Partition s of a row leaves (o_s, m_s, l_s): the unnormalised output over
// its keys, its reference max and its sum of exponentials, m_s in log2 units
// of the scaled score. With M = max_s m_s and w_s = 2^(m_s - M):
//   L = sum_s w_s l_s,  O = (sum_s w_s o_s) / L,  lse = (M + log2 L) ln 2.
// This is the rescaling of "IO-Aware Attention: Tiling the Score Matrix
// Without Materializing It", section "Parallelism and the cost of the
// split": each partition's partial output and normaliser, combined exactly.
// A partition that saw no key has m_s = -inf and weight 0; a row with no key
// at all (L = 0) gets O = 0 and lse = -inf.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace merge {

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// One warp merges one row: `part` points at the row's S partials
// ([S][d + 4] floats), `orow` at its d 16-bit outputs, `lse_row` at its lse.
// Lane i owns dims [i*d/32, (i+1)*d/32). Partials are read through L2
// (ld.global.cg): the fused merge reads what other SMs wrote in the same
// grid. The o loads of up to 16 partitions are issued before their FMAs.
template <int D, bool BF16>
__device__ __forceinline__ void merge_row(const float* __restrict__ part, int S,
                                          uint8_t* __restrict__ orow, float* __restrict__ lse_row,
                                          int lane) {
  constexpr int PER = D / 32;  // dims per lane: 2 or 4
  constexpr size_t stride = decode_partial_floats(D);
  // each lane reads (m, l) of partitions lane, lane + 32, ...
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldcg(part + s * stride + D));
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, w));
  float L = 0.f;
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int s0 = 0; s0 < S; s0 += 32) {
    const int s_mine = s0 + lane;
    float w_mine = 0.f;
    if (s_mine < S) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(part + s_mine * stride + D));
      w_mine = (ml.x == -INFINITY) ? 0.f : ex2_approx(ml.x - M);
      L = fmaf(w_mine, ml.y, L);
    }
    const int n = min(32, S - s0);
    for (int t0 = 0; t0 < n; t0 += 16) {
      // up to 16 partitions' o loads in flight, then their FMAs
      float v[16][PER];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        if (t0 + t < n) {
          const float* ps = part + (s0 + t0 + t) * stride + lane * PER;
          if constexpr (PER == 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(ps));
            v[t][0] = x.x; v[t][1] = x.y; v[t][2] = x.z; v[t][3] = x.w;
          } else {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(ps));
            v[t][0] = x.x; v[t][1] = x.y;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        // weights broadcast from the lane that computed them (every lane
        // takes part in the shuffle; lanes past n contribute nothing)
        const float w = __shfl_sync(0xffffffffu, w_mine, (t0 + t) & 31);
        if (t0 + t < n) {
#pragma unroll
          for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, v[t][i], acc[i]);
        }
      }
    }
  }
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) L += __shfl_xor_sync(0xffffffffu, L, w);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint8_t* op = orow + lane * PER * 2;
  if constexpr (PER == 2) {
    *reinterpret_cast<uint32_t*>(op) = pack2<BF16>(acc[0] * inv, acc[1] * inv);
  } else {
    *reinterpret_cast<uint2*>(op) =
        make_uint2(pack2<BF16>(acc[0] * inv, acc[1] * inv), pack2<BF16>(acc[2] * inv, acc[3] * inv));
  }
  if (lane == 0) *lse_row = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace merge
}  // namespace attn
