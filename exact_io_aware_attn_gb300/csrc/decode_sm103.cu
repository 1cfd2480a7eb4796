// decode_sm103.cu -- one query row per (batch, head) against a long KV cache.
//
// Decode is a bandwidth-bound streaming reduction over the cached keys and
// values ("IO-Aware Attention: Tiling the Score Matrix Without
// Materializing It", section "Where the approach stops helping": with one
// query row the cost is reading the cache). It is not a dense contraction,
// so it runs on the CUDA cores with 128-bit coalesced loads, not on tensor
// cores.
//
// To use the whole chip when B*h is small, the keys of each (b, h) are cut
// into S partitions ("Parallelism and the cost of the split": each of P key
// partitions produces a partial output and a partial normaliser, combined
// with the same rescaling by a second kernel):
//
//   decode_split_1head_kernel  grid B*h*S: partition s of (b, h) streams
//                          its keys once, keeps the online-softmax state
//                          (m, l, o) in fp32 and writes it to the workspace
//                          (8 resident CTAs per SM).
//   decode_split_kernel<G = 2>  grouped-query heads in pairs: every cached
//                          row is read once for both query heads (groups of
//                          4 or more run on the tensor cores instead).
//   decode_paged_split_kernel  the same loop with keys gathered through a
//                          block table (paged cache, per-sequence lengths).
//   decode_combine_kernel  one warp per (b, h): M = max m_s,
//                          w_s = 2^(m_s - M), L = sum w_s l_s,
//                          O = sum w_s o_s / L, lse = (M + log2 L) ln 2;
//                          launched as a programmatic dependent of the split
//                          kernel, so its launch overlaps the split's tail.
//
// Inside a partition, groups of d/8 threads share one key (each thread owns
// 8 of the d dimensions, one 16-byte load); a warp reads consecutive keys,
// so every warp-wide load is one contiguous 512-byte segment.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "attn_status.h"
#include "merge_sm103.cuh"

namespace attn {

namespace {

constexpr int kDecThreads = 128;  // 4 warps
constexpr int kUnroll = 4;        // keys in flight per thread (x2 loads: K and V)

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      // bf16 -> fp32 is a 16-bit shift
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

// Merge (m2, l2, o2) into (m, l, o); -inf maxima carry weight 0.
template <int N>
__device__ __forceinline__ void merge_state(float& m, float& l, float (&o)[N], float m2, float l2,
                                            const float (&o2)[N]) {
  const float mn = fmaxf(m, m2);
  const float ref = (mn == -INFINITY) ? 0.f : mn;
  const float a = ex2f(m - ref);
  const float b = ex2f(m2 - ref);
  l = l * a + l2 * b;
#pragma unroll
  for (int i = 0; i < N; ++i) o[i] = o[i] * a + o2[i] * b;
  m = mn;
}

// One CTA: partition s of the keys of one query head (one query head per
// CTA: plain attention, or a grouped-query group of odd size).
// Occupancy: measured on GB300 (16K-key cache, 1.61 GB), 8 resident CTAs per
// SM stream the cache ~7% faster than the 9 that 50 registers would allow
// (230 vs 248 us at every split count tried); the bound lets the compiler
// use up to 64 registers and so fixes 8.
template <int D, bool BF16>
__global__ void __launch_bounds__(kDecThreads, 8)
    decode_split_1head_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ k,
                              const uint8_t* __restrict__ v, float* __restrict__ ws, int T_kv,
                              int S, int chunk, float scale_log2, int group) {
  constexpr int TPK = D / 8;            // threads per key
  constexpr int KPW = 32 / TPK;         // keys per warp per load
  constexpr int SLOTS = (kDecThreads / 32) * KPW;
  constexpr int ROW = D * 2;            // bytes per key row

  const int s = static_cast<int>(blockIdx.x % static_cast<unsigned>(S));
  const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(S));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPK;           // which 8 dims
  const int slot = warp * KPW + lane / TPK;

  const int lo = s * chunk;
  const int hi = min(lo + chunk, T_kv);

  float qf[8];
  unpack8<BF16>(*reinterpret_cast<const uint4*>(q + static_cast<size_t>(bh) * ROW + sub * 16), qf);
#pragma unroll
  for (int i = 0; i < 8; ++i) qf[i] *= scale_log2;

  // key/value head of this query head: with h_q = group * h_kv,
  // (b * h_q + i) / group = b * h_kv + i / group (group = 1: plain attention)
  const int kvbh = bh / group;
  const uint8_t* kp = k + static_cast<size_t>(kvbh) * T_kv * ROW + sub * 16;
  const uint8_t* vp = v + static_cast<size_t>(kvbh) * T_kv * ROW + sub * 16;

  float m = -INFINITY, l = 0.f;
  float o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = 0.f;

  for (int base = lo; base < hi; base += SLOTS * kUnroll) {
    uint4 kr[kUnroll], vr[kUnroll];
    bool valid[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int key = base + u * SLOTS + slot;
      valid[u] = key < hi;
      if (valid[u]) {
        kr[u] = ld_stream(kp + static_cast<size_t>(key) * ROW);
        vr[u] = ld_stream(vp + static_cast<size_t>(key) * ROW);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float sc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float kf[8];
      unpack8<BF16>(kr[u], kf);
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
#pragma unroll
      for (int w = 1; w < TPK; w <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
      sc[u] = valid[u] ? dot : -INFINITY;
    }
    float mt = m;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) mt = fmaxf(mt, sc[u]);
    const float ref = (mt == -INFINITY) ? 0.f : mt;
    const float a = ex2f(m - ref);
    l *= a;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] *= a;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float p = ex2f(sc[u] - ref);
      l += p;
      float vf[8];
      unpack8<BF16>(vr[u], vf);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[i], o[i]);
    }
    m = mt;
  }

  // Merge the key slots of this warp (lanes with the same `sub`).
#pragma unroll
  for (int w = TPK; w < 32; w <<= 1) {
    float o2[8];
    const float m2 = __shfl_xor_sync(0xffffffffu, m, w);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) o2[i] = __shfl_xor_sync(0xffffffffu, o[i], w);
    merge_state<8>(m, l, o, m2, l2, o2);
  }
  // Then the four warps.
  __shared__ float sh_o[4][D];
  __shared__ float sh_ml[4][2];
  if (lane < TPK) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sh_o[warp][sub * 8 + i] = o[i];
    if (lane == 0) {
      sh_ml[warp][0] = m;
      sh_ml[warp][1] = l;
    }
  }
  __syncthreads();
  if (warp == 0 && lane < TPK) {
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      float o2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o2[i] = sh_o[w][sub * 8 + i];
      merge_state<8>(m, l, o, sh_ml[w][0], sh_ml[w][1], o2);
    }
    float* part = ws + (static_cast<size_t>(bh) * S + s) * decode_partial_floats(D);
    *reinterpret_cast<float4*>(part + sub * 8) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(part + sub * 8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    if (lane == 0) *reinterpret_cast<float4*>(part + D) = make_float4(m, l, 0.f, 0.f);
  }
  // The merge kernel is launched as a programmatic dependent of this grid:
  // once every CTA has passed this point (or exited) it may be scheduled, and
  // it waits (griddepcontrol.wait) for this grid's completion and memory
  // flush before reading any partial.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One CTA: partition s of the keys of one query head of one sequence, with
// the cache in pages: key t of sequence b is row t % page_size of page
// block_table[b][t / page_size]; a page holds page_size rows of every
// key/value head ([num_pages][h_kv][page_size][d]). Each sequence has its
// own length (seq_lens[b], clamped to the pages its table can name) and is
// cut into S partitions of ceil(len / S) keys. A table entry outside the
// pool is never dereferenced: the key is skipped and ATTN_ERR_INVALID_ARG is
// recorded in the status word (first error wins).
template <int D, bool BF16>
__global__ void __launch_bounds__(kDecThreads)
    decode_paged_split_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ kpg,
                              const uint8_t* __restrict__ vpg, const int* __restrict__ table,
                              const int* __restrict__ lens, float* __restrict__ ws, int S,
                              float scale_log2, int h_q, int group, int h_kv, int page_shift,
                              int max_pages, int num_pages, unsigned int* __restrict__ status) {
  constexpr int TPK = D / 8;            // threads per key
  constexpr int KPW = 32 / TPK;         // keys per warp per load
  constexpr int SLOTS = (kDecThreads / 32) * KPW;
  constexpr int ROW = D * 2;            // bytes per key row

  const int s = static_cast<int>(blockIdx.x % static_cast<unsigned>(S));
  const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(S));  // b * h_q + head
  const int b = bh / h_q;
  const int kvh = (bh - b * h_q) / group;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPK;           // which 8 dims
  const int slot = warp * KPW + lane / TPK;

  const int len = max(0, min(__ldg(lens + b), max_pages << page_shift));
  const int chunk = (len + S - 1) / S;
  const int lo = min(s * chunk, len);
  const int hi = min(lo + chunk, len);
  const int* trow = table + static_cast<size_t>(b) * max_pages;
  const int row_mask = (1 << page_shift) - 1;
  // rows of one page across all heads, and this head's first row in a page
  const size_t page_rows = static_cast<size_t>(h_kv) << page_shift;
  const uint8_t* kbase = kpg + (static_cast<size_t>(kvh) << page_shift) * ROW + sub * 16;
  const uint8_t* vbase = vpg + (static_cast<size_t>(kvh) << page_shift) * ROW + sub * 16;

  float qf[8];
  unpack8<BF16>(*reinterpret_cast<const uint4*>(q + static_cast<size_t>(bh) * ROW + sub * 16), qf);
#pragma unroll
  for (int i = 0; i < 8; ++i) qf[i] *= scale_log2;

  float m = -INFINITY, l = 0.f;
  float o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = 0.f;

  for (int base = lo; base < hi; base += SLOTS * kUnroll) {
    uint4 kr[kUnroll], vr[kUnroll];
    bool valid[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int key = base + u * SLOTS + slot;
      valid[u] = key < hi;
      kr[u] = make_uint4(0, 0, 0, 0);
      vr[u] = make_uint4(0, 0, 0, 0);
      if (valid[u]) {
        const int pg = __ldg(trow + (key >> page_shift));
        if (static_cast<unsigned>(pg) < static_cast<unsigned>(num_pages)) {
          const size_t off = (static_cast<size_t>(pg) * page_rows + (key & row_mask)) * ROW;
          kr[u] = ld_stream(kbase + off);
          vr[u] = ld_stream(vbase + off);
        } else {
          valid[u] = false;
          atomicCAS(status, 0u, status_word_code(1u /* ATTN_ERR_INVALID_ARG */, kKernDecodePaged, 1u));
        }
      }
    }
    float sc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float kf[8];
      unpack8<BF16>(kr[u], kf);
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
#pragma unroll
      for (int w = 1; w < TPK; w <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
      sc[u] = valid[u] ? dot : -INFINITY;
    }
    float mt = m;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) mt = fmaxf(mt, sc[u]);
    const float ref = (mt == -INFINITY) ? 0.f : mt;
    const float a = ex2f(m - ref);
    l *= a;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] *= a;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float p = ex2f(sc[u] - ref);
      l += p;
      float vf[8];
      unpack8<BF16>(vr[u], vf);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[i], o[i]);
    }
    m = mt;
  }

  // Merge the key slots of this warp (lanes with the same `sub`).
#pragma unroll
  for (int w = TPK; w < 32; w <<= 1) {
    float o2[8];
    const float m2 = __shfl_xor_sync(0xffffffffu, m, w);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) o2[i] = __shfl_xor_sync(0xffffffffu, o[i], w);
    merge_state<8>(m, l, o, m2, l2, o2);
  }
  // Then the four warps.
  __shared__ float sh_o[4][D];
  __shared__ float sh_ml[4][2];
  if (lane < TPK) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sh_o[warp][sub * 8 + i] = o[i];
    if (lane == 0) {
      sh_ml[warp][0] = m;
      sh_ml[warp][1] = l;
    }
  }
  __syncthreads();
  if (warp == 0 && lane < TPK) {
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      float o2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o2[i] = sh_o[w][sub * 8 + i];
      merge_state<8>(m, l, o, sh_ml[w][0], sh_ml[w][1], o2);
    }
    float* part = ws + (static_cast<size_t>(bh) * S + s) * decode_partial_floats(D);
    *reinterpret_cast<float4*>(part + sub * 8) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(part + sub * 8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    if (lane == 0) *reinterpret_cast<float4*>(part + D) = make_float4(m, l, 0.f, 0.f);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One CTA: partition s of the keys of one key/value head, for G query heads
// that share it (grouped-query attention with an even group below 4; groups
// of 4 or more decode on the tensor cores). Every cached key and value row is
// read once and used for all G heads. Measured on GB300: at G = 4 and 8 the
// 2*d*G FMAs and G dot-product shuffle trees per cached key leave the kernel
// issue-bound (59% and 17% of HBM at d = 128), which is why larger groups
// take the tensor-core path.
template <int D, bool BF16, int G>
__global__ void __launch_bounds__(kDecThreads)
    decode_split_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ k,
                        const uint8_t* __restrict__ v, float* __restrict__ ws, int T_kv, int S,
                        int chunk, float scale_log2, int h_q, int h_kv) {
  constexpr int TPK = D / 8;            // threads per key
  constexpr int KPW = 32 / TPK;         // keys per warp per load
  constexpr int SLOTS = (kDecThreads / 32) * KPW;
  constexpr int ROW = D * 2;            // bytes per key row
  constexpr int UNR = (G >= 4) ? 2 : kUnroll;  // keys in flight per thread (registers)

  const int s = static_cast<int>(blockIdx.x % static_cast<unsigned>(S));
  const int grp = static_cast<int>(blockIdx.x / static_cast<unsigned>(S));
  const int group = h_q / h_kv;
  const int n_sub = group / G;          // CTAs sharing one key/value head
  const int kvbh = grp / n_sub;         // b * h_kv + key/value head
  const int b = kvbh / h_kv;
  const int hq0 = (kvbh % h_kv) * group + (grp % n_sub) * G;  // first query head
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPK;           // which 8 dims
  const int slot = warp * KPW + lane / TPK;

  const int lo = s * chunk;
  const int hi = min(lo + chunk, T_kv);

  float qf[G][8];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const size_t bhq = static_cast<size_t>(b) * h_q + hq0 + i;
    unpack8<BF16>(*reinterpret_cast<const uint4*>(q + bhq * ROW + sub * 16), qf[i]);
#pragma unroll
    for (int t = 0; t < 8; ++t) qf[i][t] *= scale_log2;
  }

  const uint8_t* kp = k + static_cast<size_t>(kvbh) * T_kv * ROW + sub * 16;
  const uint8_t* vp = v + static_cast<size_t>(kvbh) * T_kv * ROW + sub * 16;

  float m[G], l[G], o[G][8];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) o[i][t] = 0.f;
  }

  for (int base = lo; base < hi; base += SLOTS * UNR) {
    uint4 kr[UNR], vr[UNR];
    bool valid[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int key = base + u * SLOTS + slot;
      valid[u] = key < hi;
      if (valid[u]) {
        kr[u] = ld_stream(kp + static_cast<size_t>(key) * ROW);
        vr[u] = ld_stream(vp + static_cast<size_t>(key) * ROW);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float sc[UNR][G];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float kf[8];
      unpack8<BF16>(kr[u], kf);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float dot = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) dot = fmaf(qf[i][t], kf[t], dot);
#pragma unroll
        for (int w = 1; w < TPK; w <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
        sc[u][i] = valid[u] ? dot : -INFINITY;
      }
    }
    // unpack each value row once for all G heads
    float vf[UNR][8];
#pragma unroll
    for (int u = 0; u < UNR; ++u) unpack8<BF16>(vr[u], vf[u]);
#pragma unroll
    for (int i = 0; i < G; ++i) {
      float mt = m[i];
#pragma unroll
      for (int u = 0; u < UNR; ++u) mt = fmaxf(mt, sc[u][i]);
      const float ref = (mt == -INFINITY) ? 0.f : mt;
      const float a = ex2f(m[i] - ref);
      l[i] *= a;
#pragma unroll
      for (int t = 0; t < 8; ++t) o[i][t] *= a;
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const float pr = ex2f(sc[u][i] - ref);
        l[i] += pr;
#pragma unroll
        for (int t = 0; t < 8; ++t) o[i][t] = fmaf(pr, vf[u][t], o[i][t]);
      }
      m[i] = mt;
    }
  }

  // Merge the key slots of this warp (lanes with the same `sub`), head by head.
#pragma unroll
  for (int i = 0; i < G; ++i) {
#pragma unroll
    for (int w = TPK; w < 32; w <<= 1) {
      float o2[8];
      const float m2 = __shfl_xor_sync(0xffffffffu, m[i], w);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[i], w);
#pragma unroll
      for (int t = 0; t < 8; ++t) o2[t] = __shfl_xor_sync(0xffffffffu, o[i][t], w);
      merge_state<8>(m[i], l[i], o[i], m2, l2, o2);
    }
  }
  // Then the four warps.
  __shared__ float sh_o[4][G][D];
  __shared__ float sh_ml[4][G][2];
  if (lane < TPK) {
#pragma unroll
    for (int i = 0; i < G; ++i) {
#pragma unroll
      for (int t = 0; t < 8; ++t) sh_o[warp][i][sub * 8 + t] = o[i][t];
      if (lane == 0) {
        sh_ml[warp][i][0] = m[i];
        sh_ml[warp][i][1] = l[i];
      }
    }
  }
  __syncthreads();
  if (warp == 0 && lane < TPK) {
#pragma unroll
    for (int i = 0; i < G; ++i) {
#pragma unroll
      for (int w = 1; w < 4; ++w) {
        float o2[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) o2[t] = sh_o[w][i][sub * 8 + t];
        merge_state<8>(m[i], l[i], o[i], sh_ml[w][i][0], sh_ml[w][i][1], o2);
      }
      const size_t bhq = static_cast<size_t>(b) * h_q + hq0 + i;
      float* part = ws + (bhq * S + s) * decode_partial_floats(D);
      *reinterpret_cast<float4*>(part + sub * 8) = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
      *reinterpret_cast<float4*>(part + sub * 8 + 4) =
          make_float4(o[i][4], o[i][5], o[i][6], o[i][7]);
      if (lane == 0) *reinterpret_cast<float4*>(part + D) = make_float4(m[i], l[i], 0.f, 0.f);
    }
  }
  // The merge kernel is launched as a programmatic dependent of this grid:
  // once every CTA has passed this point (or exited) it may be scheduled, and
  // it waits (griddepcontrol.wait) for this grid's completion and memory
  // flush before reading any partial.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int D, bool BF16>
__global__ void __launch_bounds__(128)
    decode_combine_kernel(const float* __restrict__ ws, uint8_t* __restrict__ out,
                          float* __restrict__ lse, int BH, int S) {
  // wait for the split grid (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x * 4 + warp;
  if (bh >= BH) return;
  merge::merge_row<D, BF16>(ws + static_cast<size_t>(bh) * S * decode_partial_floats(D), S,
                            out + static_cast<size_t>(bh) * D * 2, lse + bh, lane);
}

template <int D, bool BF16, int G>
cudaError_t launch_t(const FwdProblem& p, int S, float* ws, cudaStream_t stream) {
  const int BH = p.B * p.h;
  const long long rows = static_cast<long long>(p.B) * p.h_kv * ((p.h / p.h_kv) / G);
  const int chunk = (p.T_kv + S - 1) / S;
  const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
  dim3 g1(static_cast<unsigned>(S) * static_cast<unsigned>(rows));
  if constexpr (G == 1) {
    decode_split_1head_kernel<D, BF16><<<g1, kDecThreads, 0, stream>>>(
        static_cast<const uint8_t*>(p.q), static_cast<const uint8_t*>(p.k),
        static_cast<const uint8_t*>(p.v), ws, p.T_kv, S, chunk, scale_log2, p.h / p.h_kv);
  } else {
    decode_split_kernel<D, BF16, G><<<g1, kDecThreads, 0, stream>>>(
        static_cast<const uint8_t*>(p.q), static_cast<const uint8_t*>(p.k),
        static_cast<const uint8_t*>(p.v), ws, p.T_kv, S, chunk, scale_log2, p.h, p.h_kv);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the merge is a programmatic dependent launch: it may start while the
  // split grid drains and waits for it on the device (griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((BH + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, BF16>, static_cast<const float*>(ws),
                            static_cast<uint8_t*>(p.o), p.lse, BH, S);
}

template <int D, bool BF16>
cudaError_t launch_g(const FwdProblem& p, int S, float* ws, cudaStream_t stream) {
  switch (decode_heads_per_cta(p.h / p.h_kv)) {
    case 2: return launch_t<D, BF16, 2>(p, S, ws, stream);
    default: return launch_t<D, BF16, 1>(p, S, ws, stream);
  }
}

template <int D, bool BF16>
cudaError_t launch_paged_t(const PagedProblem& p, int S, float* ws, cudaStream_t stream) {
  const int BH = p.B * p.h_q;
  const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
  dim3 g1(static_cast<unsigned>(S) * static_cast<unsigned>(BH));
  decode_paged_split_kernel<D, BF16><<<g1, kDecThreads, 0, stream>>>(
      static_cast<const uint8_t*>(p.q), static_cast<const uint8_t*>(p.k_pages),
      static_cast<const uint8_t*>(p.v_pages), p.block_table, p.seq_lens, ws, S, scale_log2, p.h_q,
      p.h_q / p.h_kv, p.h_kv, p.page_shift, p.max_pages, p.num_pages, p.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((BH + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, BF16>, static_cast<const float*>(ws),
                            static_cast<uint8_t*>(p.o), p.lse, BH, S);
}

}  // namespace

cudaError_t launch_decode(const FwdProblem& p, int num_splits, float* ws, cudaStream_t stream,
                          const char** name) {
  cudaError_t e;
  const bool gqa = p.h_kv != p.h;
  if (p.d == 64) {
    e = p.bf16 ? launch_g<64, true>(p, num_splits, ws, stream)
               : launch_g<64, false>(p, num_splits, ws, stream);
    *name = gqa ? (p.bf16 ? "decode_split_gqa_d64_bf16+decode_combine"
                          : "decode_split_gqa_d64_f16+decode_combine")
                : (p.bf16 ? "decode_split_d64_bf16+decode_combine"
                          : "decode_split_d64_f16+decode_combine");
  } else {
    e = p.bf16 ? launch_g<128, true>(p, num_splits, ws, stream)
               : launch_g<128, false>(p, num_splits, ws, stream);
    *name = gqa ? (p.bf16 ? "decode_split_gqa_d128_bf16+decode_combine"
                          : "decode_split_gqa_d128_f16+decode_combine")
                : (p.bf16 ? "decode_split_d128_bf16+decode_combine"
                          : "decode_split_d128_f16+decode_combine");
  }
  return e;
}

int decode_split_ctas_per_sm(int d, int heads_per_cta) {
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  const size_t smem = 0;
  auto occ = [&](auto kern) { return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecThreads, smem); };
  if (d == 64) {
    switch (heads_per_cta) {
      case 2: e = occ(decode_split_kernel<64, true, 2>); break;
      default: e = occ(decode_split_1head_kernel<64, true>); break;
    }
  } else {
    switch (heads_per_cta) {
      case 2: e = occ(decode_split_kernel<128, true, 2>); break;
      default: e = occ(decode_split_1head_kernel<128, true>); break;
    }
  }
  return (e == cudaSuccess && n > 0) ? n : 8;
}

}  // namespace attn

namespace attn {

cudaError_t launch_decode_paged(const PagedProblem& p, int num_splits, float* ws,
                                cudaStream_t stream, const char** name) {
  cudaError_t e;
  if (p.d == 64) {
    e = p.bf16 ? launch_paged_t<64, true>(p, num_splits, ws, stream)
               : launch_paged_t<64, false>(p, num_splits, ws, stream);
    *name = p.bf16 ? "decode_paged_split_d64_bf16+decode_combine"
                   : "decode_paged_split_d64_f16+decode_combine";
  } else {
    e = p.bf16 ? launch_paged_t<128, true>(p, num_splits, ws, stream)
               : launch_paged_t<128, false>(p, num_splits, ws, stream);
    *name = p.bf16 ? "decode_paged_split_d128_bf16+decode_combine"
                   : "decode_paged_split_d128_f16+decode_combine";
  }
  return e;
}

cudaError_t launch_combine(const float* part, void* o, float* lse, long long rows, int S, int d,
                           bool bf16, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int n = static_cast<int>(rows);
  uint8_t* out = static_cast<uint8_t*>(o);
  if (d == 64)
    return bf16 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<64, true>, part, out, lse, n, S)
                : cudaLaunchKernelEx(&cfg, decode_combine_kernel<64, false>, part, out, lse, n, S);
  return bf16 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<128, true>, part, out, lse, n, S)
              : cudaLaunchKernelEx(&cfg, decode_combine_kernel<128, false>, part, out, lse, n, S);
}

int decode_paged_ctas_per_sm(int d) {
  int n = 0;
  const cudaError_t e =
      d == 64 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_paged_split_kernel<64, true>,
                                                              kDecThreads, 0)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_paged_split_kernel<128, true>,
                                                              kDecThreads, 0);
  return (e == cudaSuccess && n > 0) ? n : 8;
}

}  // namespace attn
