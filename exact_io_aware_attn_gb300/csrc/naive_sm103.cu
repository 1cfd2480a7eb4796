// naive_sm103.cu -- the materialising attention the IO-aware kernels are
// measured against: the whole score matrix S and probability matrix P are
// written to HBM, as "Attention and Its Computational Cost" describes for
// the standard implementation (section "The cost of writing down the
// scores": one T x T score tensor per head, then softmax, then P V) and as
// "E8.1 IO-aware attention" Part 2 writes standard_attention.
//
// Three kernels, one per step of that definition:
//   naive_scores_kernel   S = scale * Q K^T (masked entries -inf), 16-bit,
//                         [B*h][T_q][T_kv]
//   naive_softmax_kernel  per row: m = max, l = sum exp(s - m),
//                         P = exp(s - m) / l (16-bit), lse = m + ln l
//   naive_pv_kernel       O = P V, 16-bit
// The two products use warp-level mma.sync (m16n8k16, fp32 accumulate) from
// shared-memory tiles; the softmax is one warp per row. This path exists to
// be timed and measured beside the IO-aware kernels (its traffic is the
// 2 x T_q x T_kv 16-bit matrices written and read back); it is not tuned.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kTile = 128;      // query rows (and keys) per score tile
constexpr int kPvKeys = 64;     // keys per step of the P V product
constexpr int kNaiveThreads = 256;

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}

template <bool BF16>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

template <bool BF16>
__device__ __forceinline__ float from16(uint16_t x) {
  if constexpr (BF16) return __bfloat162float(__ushort_as_bfloat16(x));
  else return __half2float(__ushort_as_half(x));
}

__device__ __forceinline__ uint32_t lds32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// Copies rows [r0, r0 + 128) of a [rows][D] 16-bit matrix into shared memory
// with row stride D + 8 (conflict-free fragment loads); rows past `rows`
// read as zero.
template <int D>
__device__ __forceinline__ void load_tile(uint16_t* dst, const uint16_t* src, int r0, int rows) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  for (int i = threadIdx.x; i < kTile * CH; i += kNaiveThreads) {
    const int r = i / CH, c = (i % CH) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < rows) v = *reinterpret_cast<const uint4*>(src + (static_cast<size_t>(r0 + r) * D + c));
    uint32_t* d = reinterpret_cast<uint32_t*>(dst + r * (D + 8) + c);
    d[0] = v.x;
    d[1] = v.y;
    d[2] = v.z;
    d[3] = v.w;
  }
}

// S tile (128 query rows x 128 keys) of one head. 8 warps: warp w computes
// rows [32 (w % 4), +32) x keys [64 (w / 4), +64).
template <int D, bool BF16>
__global__ void __launch_bounds__(kNaiveThreads)
    naive_scores_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                        uint16_t* __restrict__ s, int T_q, int T_kv, float scale, int causal) {
  extern __shared__ uint16_t sm[];
  uint16_t* qs = sm;
  uint16_t* ks = sm + kTile * (D + 8);
  const int bh = blockIdx.z;
  const int i0 = blockIdx.y * kTile, j0 = blockIdx.x * kTile;
  load_tile<D>(qs, q + static_cast<size_t>(bh) * T_q * D, i0, T_q);
  load_tile<D>(ks, k + static_cast<size_t>(bh) * T_kv * D, j0, T_kv);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int m0 = (warp & 3) * 32, n0 = (warp >> 2) * 64;
  float acc[2][8][4] = {};
#pragma unroll
  for (int kk = 0; kk < D; kk += 16) {
    uint32_t a[2][4], b[8][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const uint16_t* r = qs + (m0 + mt * 16 + g) * (D + 8) + kk + t * 2;
      a[mt][0] = lds32(r);
      a[mt][1] = lds32(r + 8 * (D + 8));
      a[mt][2] = lds32(r + 8);
      a[mt][3] = lds32(r + 8 * (D + 8) + 8);
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const uint16_t* r = ks + (n0 + nt * 8 + g) * (D + 8) + kk + t * 2;
      b[nt][0] = lds32(r);
      b[nt][1] = lds32(r + 8);
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) mma16816<BF16>(acc[mt][nt], a[mt], b[nt]);
  }
  const int off = T_kv - T_q;  // bottom-right causal alignment
  uint16_t* sh = s + static_cast<size_t>(bh) * T_q * T_kv;
  const bool pairs = (T_kv & 1) == 0;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = i0 + m0 + mt * 16 + g + half * 8;
      if (row >= T_q) continue;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int key = j0 + n0 + nt * 8 + t * 2;
        if (key >= T_kv) continue;
        float v0 = acc[mt][nt][2 * half] * scale, v1 = acc[mt][nt][2 * half + 1] * scale;
        if (causal && key > row + off) v0 = -INFINITY;
        if (causal && key + 1 > row + off) v1 = -INFINITY;
        uint16_t* dst = sh + static_cast<size_t>(row) * T_kv + key;
        if (pairs) {
          *reinterpret_cast<uint32_t*>(dst) =
              static_cast<uint32_t>(to16<BF16>(v0)) | (static_cast<uint32_t>(to16<BF16>(v1)) << 16);
        } else {
          dst[0] = to16<BF16>(v0);
          if (key + 1 < T_kv) dst[1] = to16<BF16>(v1);
        }
      }
    }
}

// One warp per row of S. First pass: the row's max and sum of exponentials
// in one read (each lane keeps a running max and a sum rescaled when its max
// grows; the lanes' pairs are then merged). Second pass: P = exp(s - m) / l
// written as 16-bit.
template <bool BF16>
__global__ void __launch_bounds__(kNaiveThreads)
    naive_softmax_kernel(const uint16_t* __restrict__ s, uint16_t* __restrict__ p,
                         float* __restrict__ lse, long long rows, int T_kv) {
  const long long row = static_cast<long long>(blockIdx.x) * (kNaiveThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const uint16_t* sr = s + static_cast<size_t>(row) * T_kv;
  uint16_t* pr = p + static_cast<size_t>(row) * T_kv;
  const bool vec = (T_kv & 7) == 0;  // rows start on 16-byte boundaries
  float m = -INFINITY, l = 0.f;
  auto take = [&](float x) {
    if (x > m) {
      l = l * __expf(m - x) + 1.f;  // exp(-inf) = 0 on the first finite value
      m = x;
    } else if (x != -INFINITY) {  // a masked score adds nothing
      l += __expf(x - m);
    }
  };
  if (vec) {
    for (int c = lane * 8; c < T_kv; c += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(sr + c);
      const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
      for (int i = 0; i < 8; ++i) take(from16<BF16>(e[i]));
    }
  } else {
    for (int c = lane; c < T_kv; c += 32) take(from16<BF16>(sr[c]));
  }
  // merge the lanes' (m, l)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, m2);
    l = (mn == -INFINITY) ? 0.f : l * __expf(m - mn) + l2 * __expf(m2 - mn);
    m = mn;
  }
  const float inv = 1.f / l;
  if (vec) {
    for (int c = lane * 8; c < T_kv; c += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(sr + c);
      const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
      uint4 w;
      uint16_t* o = reinterpret_cast<uint16_t*>(&w);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = to16<BF16>(__expf(from16<BF16>(e[i]) - m) * inv);
      *reinterpret_cast<uint4*>(pr + c) = w;
    }
  } else {
    for (int c = lane; c < T_kv; c += 32) pr[c] = to16<BF16>(__expf(from16<BF16>(sr[c]) - m) * inv);
  }
  if (lane == 0) lse[row] = m + logf(l);
}

// O tile (128 query rows x D) of one head. 8 warps: warp w owns rows
// [16 w, 16 w + 16). Per step of 64 keys the P tile is staged row-major and
// the V tile transposed ([D][keys]) in shared memory; the next step's tiles
// are fetched into registers while this step's products run.
template <int D, bool BF16>
__global__ void __launch_bounds__(kNaiveThreads)
    naive_pv_kernel(const uint16_t* __restrict__ p, const uint16_t* __restrict__ v,
                    uint16_t* __restrict__ o, int T_q, int T_kv) {
  constexpr int PS = kPvKeys + 8;                            // staged row stride (elements)
  constexpr int PCH = kTile * kPvKeys / 8 / kNaiveThreads;   // 16-byte P chunks per thread
  constexpr int VCH = kPvKeys * D / 8 / kNaiveThreads;       // 16-byte V chunks per thread
  __shared__ __align__(16) uint16_t ps[kTile * PS];
  __shared__ __align__(16) uint16_t vt[D * PS];
  const int bh = blockIdx.y;
  const int i0 = blockIdx.x * kTile;
  const uint16_t* ph = p + static_cast<size_t>(bh) * T_q * T_kv;
  const uint16_t* vh = v + static_cast<size_t>(bh) * T_kv * D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const bool vec = (T_kv & 7) == 0;  // P rows start on 16-byte boundaries
  uint4 pr[PCH], vr[VCH];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int j = 0; j < PCH; ++j) {
      const int i = threadIdx.x + j * kNaiveThreads;
      const int row = i0 + i / (kPvKeys / 8), key = k0 + (i % (kPvKeys / 8)) * 8;
      if (vec && row < T_q && key < T_kv) {
        pr[j] = *reinterpret_cast<const uint4*>(ph + static_cast<size_t>(row) * T_kv + key);
      } else {
        uint16_t* e = reinterpret_cast<uint16_t*>(&pr[j]);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          e[u] = (row < T_q && key + u < T_kv) ? ph[static_cast<size_t>(row) * T_kv + key + u] : 0;
      }
    }
#pragma unroll
    for (int j = 0; j < VCH; ++j) {
      const int i = threadIdx.x + j * kNaiveThreads;
      const int kr = i / (D / 8), c = (i % (D / 8)) * 8;
      vr[j] = make_uint4(0u, 0u, 0u, 0u);
      if (k0 + kr < T_kv) vr[j] = *reinterpret_cast<const uint4*>(vh + static_cast<size_t>(k0 + kr) * D + c);
    }
  };
  float acc[D / 8][4] = {};
  fetch(0);
  for (int k0 = 0; k0 < T_kv; k0 += kPvKeys) {
    __syncthreads();  // the previous step's products have read the tiles
#pragma unroll
    for (int j = 0; j < PCH; ++j) {
      const int i = threadIdx.x + j * kNaiveThreads;
      *reinterpret_cast<uint4*>(ps + (i / (kPvKeys / 8)) * PS + (i % (kPvKeys / 8)) * 8) = pr[j];
    }
#pragma unroll
    for (int j = 0; j < VCH; ++j) {
      const int i = threadIdx.x + j * kNaiveThreads;
      const int kr = i / (D / 8), c = (i % (D / 8)) * 8;
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(&vr[j]);
#pragma unroll
      for (int u = 0; u < 8; ++u) vt[(c + u) * PS + kr] = xs[u];
    }
    __syncthreads();
    if (k0 + kPvKeys < T_kv) fetch(k0 + kPvKeys);
#pragma unroll
    for (int ks = 0; ks < kPvKeys; ks += 16) {
      uint32_t a[4];
      const uint16_t* r = ps + (warp * 16 + g) * PS + ks + t * 2;
      a[0] = lds32(r);
      a[1] = lds32(r + 8 * PS);
      a[2] = lds32(r + 8);
      a[3] = lds32(r + 8 * PS + 8);
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        uint32_t b[2];
        const uint16_t* c = vt + (nt * 8 + g) * PS + ks + t * 2;
        b[0] = lds32(c);
        b[1] = lds32(c + 8);
        mma16816<BF16>(acc[nt], a, b);
      }
    }
  }
  uint16_t* oh = o + static_cast<size_t>(bh) * T_q * D;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = i0 + warp * 16 + g + half * 8;
    if (row >= T_q) continue;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + t * 2;
      *reinterpret_cast<uint32_t*>(oh + static_cast<size_t>(row) * D + col) =
          static_cast<uint32_t>(to16<BF16>(acc[nt][2 * half])) |
          (static_cast<uint32_t>(to16<BF16>(acc[nt][2 * half + 1])) << 16);
    }
  }
}

template <int D, bool BF16>
cudaError_t launch_naive_t(const FwdProblem& p, uint16_t* s, uint16_t* pm, cudaStream_t stream) {
  const size_t smem = 2 * kTile * (D + 8) * sizeof(uint16_t);
  static std::mutex mu;
  static uint64_t configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64 && !(configured & (1ull << dev))) {
      e = cudaFuncSetAttribute(naive_scores_kernel<D, BF16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      configured |= 1ull << dev;
    }
  }
  const int BH = p.B * p.h;
  const dim3 gs((p.T_kv + kTile - 1) / kTile, (p.T_q + kTile - 1) / kTile, BH);
  naive_scores_kernel<D, BF16><<<gs, kNaiveThreads, smem, stream>>>(
      static_cast<const uint16_t*>(p.q), static_cast<const uint16_t*>(p.k), s, p.T_q, p.T_kv,
      p.scale, p.causal);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long rows = static_cast<long long>(BH) * p.T_q;
  const long long blocks = (rows + kNaiveThreads / 32 - 1) / (kNaiveThreads / 32);
  naive_softmax_kernel<BF16><<<static_cast<unsigned>(blocks), kNaiveThreads, 0, stream>>>(
      s, pm, p.lse, rows, p.T_kv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const dim3 gp((p.T_q + kTile - 1) / kTile, BH);
  naive_pv_kernel<D, BF16><<<gp, kNaiveThreads, 0, stream>>>(pm, static_cast<const uint16_t*>(p.v),
                                                            static_cast<uint16_t*>(p.o), p.T_q, p.T_kv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_naive(const FwdProblem& p, void* workspace, cudaStream_t stream, const char** name) {
  const size_t n = static_cast<size_t>(p.B) * p.h * p.T_q * p.T_kv;
  uint16_t* s = static_cast<uint16_t*>(workspace);
  uint16_t* pm = s + n;
  cudaError_t e;
  if (p.d == 64)
    e = p.bf16 ? launch_naive_t<64, true>(p, s, pm, stream) : launch_naive_t<64, false>(p, s, pm, stream);
  else
    e = p.bf16 ? launch_naive_t<128, true>(p, s, pm, stream) : launch_naive_t<128, false>(p, s, pm, stream);
  *name = p.bf16 ? (p.d == 64 ? "naive_scores+naive_softmax+naive_pv_d64_bf16"
                              : "naive_scores+naive_softmax+naive_pv_d128_bf16")
                 : (p.d == 64 ? "naive_scores+naive_softmax+naive_pv_d64_f16"
                              : "naive_scores+naive_softmax+naive_pv_d128_f16");
  return e;
}

}  // namespace attn
