// backward_sm103.cu -- gradients of exact attention (dQ, dK, dV) on GB300
// tensor cores, by recomputation.
//
// The backward pass does not keep the probabilities: it recomputes them from
// Q, K, V and the per-row constants the forward saved (lse), one tile at a
// time, and never writes a score or probability matrix to HBM ("IO-Aware
// Attention: Tiling the Score Matrix Without Materializing It", section "What
// has to stay in fast memory"). The gradients are the derivative of the
// forward definition: with P = exp(scale * Q K^T - lse) (masked entries 0),
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D_i = rowsum(dO_i * O_i),
//   dQ = scale * dS K,  dK = scale * dS^T Q
// (D_i = sum_j P_ij dP_ij because O_i = sum_j P_ij V_j).
//
// Three launches, no atomics (so the result is deterministic):
//   bwd_prep     one pass over O and dO: D and lse * log2(e) per query row,
//                into a workspace padded to 128 rows per head
//   bwd (KV)     one CTA per (key/value head, 128-key tile): K and V stay in
//                shared memory, the CTA streams tiles of Q and dO (every
//                query head of the group, causal: only rows that see the
//                tile) and accumulates dV and dK in tensor memory. At d = 64
//                the streamed tiles have 128 rows (bwd_kv128_kernel,
//                below); at d = 128 they have 64 (bwd_kernel in KV mode)
//   bwd (Q)      one CTA per (query head, 128-row tile): Q and dO stay, the
//                CTA streams tiles of K and V (causal: up to the diagonal)
//                and accumulates dQ in tensor memory. At d = 64 the streamed
//                tiles have 128 keys (bwd_q128_kernel, below); at d = 128
//                they have 64 (bwd_kernel in Q mode)
//
// All three gradient kernels share the roles (320 threads): warps 0-7 form P
// and dS, warp 8 is the TMA producer, warp 9 owns TMEM and issues the MMAs.
//
// bwd_kernel's two modes are one template. Roles (320 threads): warps 0-7 turn
// scores into P and dS -- warp w owns TMEM lanes 32*(w%4).. (one resident row
// per thread) and columns 32*(w/4).. of each 64-column score tile, so every
// sub-partition runs two of them; warp 8 is the TMA producer; warp 9 owns TMEM
// and issues the MMAs. Per streamed tile t the tensor core computes
//   S_t  = X U_t^T and dP_t = Y W_t^T      (M=128 resident rows, N=64, K=d)
// into one of two TMEM buffers; each elementwise warp stores its 32 columns
// of P_t and dS_t as 16-bit pairs over the first 16 columns of its own half
// of S_t and dP_t (so no warp overwrites columns another warp still reads),
// and the tensor core then accumulates (A read from TMEM, B the streamed
// tile read MN-major)
//   KV mode (X=K, Y=V, U=Q, W=dO):  dV += P_t^T dO_t,  dK += dS_t^T Q_t
//   Q mode  (X=Q, Y=dO, U=K, W=V):  dQ += dS_t K_t
// The scores of tile t+1 go into the other buffer while the elementwise warps
// work on tile t. In KV mode P_t is stored and released first (its own
// barrier), so dV += P_t^T dO_t runs while the warps form dS_t; Q mode stores
// only dS_t. In KV mode the streamed rows' lse and D are per column: the
// warps read TMEM with the 16-lane shape (each thread four keys at 8 of the
// 32 columns), so a thread needs 8 columns' values, not 32. TMEM: buffers [0,128) and
// [128,256) (S then dP, 64 columns each), dV at 256, dK or dQ at 256 + d:
// 512 columns at d = 128.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "attn_status.h"
#include "ptx_sm103.cuh"
#include "tma_host.h"

namespace attn {

namespace {

constexpr int kRes = 128;              // resident rows per CTA (TMEM lanes, M of every MMA)
constexpr int kStr = 64;               // rows of one streamed tile
constexpr int kSubRes = kRes * 128;    // one [128 rows][64 x 16-bit] swizzled sub-tile
constexpr int kSubStr = kStr * 128;    // one [64 rows][64 x 16-bit] swizzled sub-tile
constexpr int kBwdThreads = 320;
constexpr int kWarpProd = 8;
constexpr int kWarpMma = 9;
constexpr int kEltThreads = 256;       // warps 0-7
constexpr uint32_t kColAcc1 = 256;     // dV (KV mode)

template <int D, bool KV>
struct BwdCfg {
  static constexpr int RES_BYTES = kRes * D * 2;           // X or Y
  static constexpr int STR_BYTES = kStr * D * 2;           // U or W
  static constexpr int VEC_BYTES = KV ? 2 * kStr * 4 : 0;  // lse*log2e and D of the streamed rows
  static constexpr int STAGE_BYTES = (2 * STR_BYTES + VEC_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGES = (D == 64) ? 6 : 4;
  static constexpr int OFF_X = 0;
  static constexpr int OFF_Y = RES_BYTES;
  static constexpr int OFF_RING = 2 * RES_BYTES;
  static constexpr int OFF_BAR = OFF_RING + STAGES * STAGE_BYTES;
  // res_full, stage_full[ST], stage_empty[ST], sp_full[2], p_full[2], acc_full, mma_done,
  // res_tmem, p_half[2]
  static constexpr int N_BARS = 1 + 2 * STAGES + 9;
  static constexpr int OFF_TMEMPTR = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_ACC2 = 256u + D;             // dK (KV mode) or dQ (Q mode)
  // The resident tiles X and Y also go to TMEM (D/2 columns each), so the
  // score products read A from TMEM and only B from shared memory -- except
  // dK/dV at d = 128, where TMEM is full (buffers 256 + dV 128 + dK 128).
  static constexpr bool XY_TMEM = !(KV && D == 128);
  static constexpr uint32_t COL_X = KV ? 256u + 2u * D : 256u;  // Q mode: the unused dV columns
  static constexpr uint32_t COL_Y = COL_X + D / 2;
};
static_assert(BwdCfg<128, false>::COL_Y + 64 <= BwdCfg<128, false>::COL_ACC2, "tensor memory");
static_assert(BwdCfg<128, true>::SMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(BwdCfg<128, false>::SMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(BwdCfg<128, true>::COL_ACC2 + 128 <= 512, "tensor memory");

__host__ __device__ constexpr uint32_t col_buf(int b) { return static_cast<uint32_t>(b) * 128u; }

enum : uint32_t {
  kSiteProdStage = 1, kSiteMmaRes, kSiteMmaStage, kSiteMmaP, kSiteEltS, kSiteEltStage, kSiteEltAcc,
  kSiteEltRes, kSiteMmaSFree
};

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

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

__device__ __forceinline__ void tmem_wait_ld_64(uint32_t (&r)[64]) {
#define R8(b) "+r"(r[b]), "+r"(r[b + 1]), "+r"(r[b + 2]), "+r"(r[b + 3]), "+r"(r[b + 4]), \
              "+r"(r[b + 5]), "+r"(r[b + 6]), "+r"(r[b + 7])
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : R8(0), R8(8), R8(16), R8(24), R8(32), R8(40), R8(48), R8(56)
               :
               : "memory");
#undef R8
}

__device__ __forceinline__ void tmem_wait_ld_32(uint32_t (&r)[32]) {
#define R8(b) "+r"(r[b]), "+r"(r[b + 1]), "+r"(r[b + 2]), "+r"(r[b + 3]), "+r"(r[b + 4]), \
              "+r"(r[b + 5]), "+r"(r[b + 6]), "+r"(r[b + 7])
  asm volatile("tcgen05.wait::ld.sync.aligned;" : R8(0), R8(8), R8(16), R8(24) : : "memory");
#undef R8
}

// Bounded wait used only while draining after an error.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = ptx::smem_u32(bar);
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(a, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// D_i = sum_c dO_ic O_ic and lse_i * log2(e), per query row, into [BH][Tq_pad]
// arrays; rows T_q..Tq_pad-1 of each head get D = 0 and +inf (so that any
// probability recomputed for them is exactly 0).
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    bwd_prep_kernel(const uint8_t* __restrict__ o, const uint8_t* __restrict__ dout,
                    const float* __restrict__ lse, float* __restrict__ l2, float* __restrict__ dd,
                    int T_q, int Tq_pad, long long n_rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 elements (16 bytes) each
  const long long row = static_cast<long long>(blockIdx.x) * (256 / TPR) + threadIdx.x / TPR;
  const int sub = threadIdx.x % TPR;
  const bool in = row < n_rows;
  const long long bh = in ? row / Tq_pad : 0;
  const int t = in ? static_cast<int>(row - bh * Tq_pad) : 0;
  const bool valid = in && t < T_q;
  float acc = 0.f;
  if (valid) {
    const size_t e = (static_cast<size_t>(bh) * T_q + t) * D + sub * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(o + e * 2);
    const uint4 g = *reinterpret_cast<const uint4*>(dout + e * 2);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = unpack2<BF16>(aw[i]), y = unpack2<BF16>(gw[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int w = 1; w < TPR; w <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
  if (in && sub == 0) {
    dd[row] = valid ? acc : 0.f;
    l2[row] = valid ? lse[static_cast<size_t>(bh) * T_q + t] * 1.4426950408889634f : INFINITY;
  }
}

// One work unit: 128 resident rows of one head and the streamed tiles it
// visits.
struct BwdUnit {
  int res_bh;    // KV: b * h_kv + key/value head; Q: b * h + query head
  int r0;        // first resident row (key in KV mode, query row in Q mode)
  int str_bh0;   // KV: first query head of the group; Q: the key/value head
  int t_first;   // KV: first streamed 64-row tile of each query head; Q: 0
  int per_head;  // streamed tiles per query head (KV) or in all (Q)
  int n_items;
};

// Units are numbered heaviest first under a causal mask: key tile 0 is seen
// by every query row, the last query tile sees the most keys.
template <bool KV>
__device__ __forceinline__ BwdUnit bwd_unit(int u, int BH_res, int n_res_tiles, int T_q, int T_kv,
                                            int causal, int h, int h_kv) {
  const int group = h / h_kv;
  const int off = T_kv - T_q;
  BwdUnit w;
  w.res_bh = u % BH_res;
  if constexpr (KV) {
    const int j = u / BH_res;
    w.r0 = j * kRes;
    const int b = w.res_bh / h_kv, kvh = w.res_bh % h_kv;
    w.str_bh0 = b * h + kvh * group;
    // key r0 is visible to query row r iff r0 <= r + off
    const int first_row = causal ? max(0, w.r0 - off) : 0;
    w.t_first = first_row / kStr;
    w.per_head = (T_q + kStr - 1) / kStr - w.t_first;
    w.n_items = w.per_head * group;
  } else {
    const int i = n_res_tiles - 1 - u / BH_res;
    w.r0 = i * kRes;
    w.str_bh0 = w.res_bh / group;  // (b * h + i) / group = b * h_kv + i / group
    w.t_first = 0;
    const int last_row = min(T_q, w.r0 + kRes) - 1;
    const int last_key = causal ? min(T_kv - 1, last_row + off) : T_kv - 1;
    w.per_head = last_key / kStr + 1;
    w.n_items = w.per_head;
  }
  return w;
}

__device__ __forceinline__ void bwd_item(const BwdUnit& w, int it, int* bh, int* s0) {
  const int g = it / w.per_head;
  *bh = w.str_bh0 + g;
  *s0 = (w.t_first + (it - g * w.per_head)) * kStr;
}

template <int D, bool BF16, bool KV>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
               const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW,
               const float* __restrict__ ws_l2, const float* __restrict__ ws_dd, int Tq_pad,
               void* __restrict__ out1, void* __restrict__ out2, int T_q, int T_kv, int BH_res,
               int n_res_tiles, int h, int h_kv, float scale, float scale_log2, int causal,
               unsigned int* __restrict__ status) {
  using C = BwdCfg<D, KV>;
  constexpr int ST = C::STAGES;
  constexpr uint32_t kKern = KV ? kKernBwdKV : kKernBwdQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* res_full = bars;
  uint64_t* stage_full = bars + 1;
  uint64_t* stage_empty = stage_full + ST;
  uint64_t* sp_full = stage_empty + ST;
  uint64_t* p_full = sp_full + 2;
  uint64_t* acc_full = p_full + 2;
  uint64_t* mma_done = acc_full + 1;
  uint64_t* res_tmem = mma_done + 1;   // X and Y copied into TMEM (XY_TMEM)
  uint64_t* p_half = res_tmem + 1;     // KV: P_t stored (dS_t still being formed)
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMPTR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const BwdUnit w =
      bwd_unit<KV>(static_cast<int>(blockIdx.x), BH_res, n_res_tiles, T_q, T_kv, causal, h, h_kv);
  const int n = w.n_items;
  const int off = T_kv - T_q;

  if (threadIdx.x == 0) {
    ptx::mbar_init(res_full, 1);
    for (int i = 0; i < ST; ++i) {
      ptx::mbar_init(&stage_full[i], 1);
      ptx::mbar_init(&stage_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sp_full[b], 1);
      ptx::mbar_init(&p_full[b], kEltThreads);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(mma_done, 1);
    ptx::mbar_init(res_tmem, kEltThreads);
    for (int b = 0; b < 2; ++b) ptx::mbar_init(&p_half[b], kEltThreads);
    ptx::fence_mbarrier_init();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(tmem_ptr, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  if (warp == kWarpProd) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmX);
      ptx::prefetch_tensormap(&tmY);
      ptx::prefetch_tensormap(&tmU);
      ptx::prefetch_tensormap(&tmW);
      // the streamed tiles are read by many CTAs (every key tile of a head,
      // or every query tile): keep them in L2; the resident ones once
      const uint64_t pol_str = ptx::policy_evict_last();
      const uint64_t pol_res = ptx::policy_evict_first();
      ptx::mbar_arrive_expect_tx(res_full, 2 * C::RES_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        ptx::tma_load_3d(smem + C::OFF_X + c * kSubRes, &tmX, res_full, c * 64, w.r0, w.res_bh,
                         pol_res);
        ptx::tma_load_3d(smem + C::OFF_Y + c * kSubRes, &tmY, res_full, c * 64, w.r0, w.res_bh,
                         pol_res);
      }
      bool ok = true;
      int it = 0;
      for (; it < n; ++it) {
        const int slot = it % ST;
        ok = ptx::mbar_wait(&stage_empty[slot], ((it / ST) & 1) ^ 1, status,
                            status_word(kKern, kSiteProdStage));
        if (!ok) break;
        int sbh, s0;
        bwd_item(w, it, &sbh, &s0);
        uint8_t* stg = smem + C::OFF_RING + slot * C::STAGE_BYTES;
        ptx::mbar_arrive_expect_tx(&stage_full[slot], 2 * C::STR_BYTES + C::VEC_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          ptx::tma_load_3d(stg + c * kSubStr, &tmU, &stage_full[slot], c * 64, s0, sbh, pol_str);
          ptx::tma_load_3d(stg + C::STR_BYTES + c * kSubStr, &tmW, &stage_full[slot], c * 64, s0,
                           sbh, pol_str);
        }
        if constexpr (KV) {
          const size_t vo = static_cast<size_t>(sbh) * Tq_pad + s0;
          ptx::bulk_load(stg + 2 * C::STR_BYTES, ws_l2 + vo, kStr * 4, &stage_full[slot]);
          ptx::bulk_load(stg + 2 * C::STR_BYTES + kStr * 4, ws_dd + vo, kStr * 4,
                         &stage_full[slot]);
        }
      }
      if (!ok) {
        // let the copies in flight land before the CTA's shared memory goes
        mbar_drain(res_full, 0);
        for (int i = (it > ST ? it - ST : 0); i < it; ++i) mbar_drain(&stage_full[i % ST], (i / ST) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs this loop in uniform control flow (so descriptor
    // arithmetic stays warp-uniform); one elected lane issues each batch of
    // MMAs and its commit. elect.sync picks the lowest active lane, the same
    // lane every time, so every commit covers that lane's earlier MMAs.
    constexpr uint32_t idS = ptx::make_idesc_f16(BF16, kRes, kStr, false, false);
    constexpr uint32_t idG = ptx::make_idesc_f16(BF16, kRes, D, false, true);
    const uint32_t sX = ptx::smem_u32(smem + C::OFF_X);
    const uint32_t sY = ptx::smem_u32(smem + C::OFF_Y);
    const uint32_t sR = ptx::smem_u32(smem + C::OFF_RING);
    // K-major views (score products) and MN-major views (gradient products)
    const uint64_t dX = ptx::make_sdesc_sw128(sX, 16, 1024);
    const uint64_t dY = ptx::make_sdesc_sw128(sY, 16, 1024);
    const uint64_t dUk = ptx::make_sdesc_sw128(sR, 16, 1024);
    const uint64_t dWk = ptx::make_sdesc_sw128(sR + C::STR_BYTES, 16, 1024);
    const uint64_t dUm = ptx::make_sdesc_sw128(sR, kSubStr, 1024);
    const uint64_t dWm = ptx::make_sdesc_sw128(sR + C::STR_BYTES, kSubStr, 1024);

    auto issue_scores = [&](int b, int slot) {
      const uint64_t so = static_cast<uint64_t>(slot * C::STAGE_BYTES) >> 4;
      const uint64_t u0 = dUk + so, w0 = dWk + so;
      const uint32_t d_s = tmem + col_buf(b);
      if (ptx::elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ro = (kk >> 2) * kSubRes + (kk & 3) * 32;
          const uint32_t to = (kk >> 2) * kSubStr + (kk & 3) * 32;
          if constexpr (C::XY_TMEM)
            ptx::mma_f16_ts(d_s, tmem + C::COL_X + kk * 8, u0 + (to >> 4), idS, kk > 0 ? 1u : 0u);
          else
            ptx::mma_f16_ss(d_s, dX + (ro >> 4), u0 + (to >> 4), idS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ro = (kk >> 2) * kSubRes + (kk & 3) * 32;
          const uint32_t to = (kk >> 2) * kSubStr + (kk & 3) * 32;
          if constexpr (C::XY_TMEM)
            ptx::mma_f16_ts(d_s + 64, tmem + C::COL_Y + kk * 8, w0 + (to >> 4), idS,
                            kk > 0 ? 1u : 0u);
          else
            ptx::mma_f16_ss(d_s + 64, dY + (ro >> 4), w0 + (to >> 4), idS, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&sp_full[b]);
      }
      __syncwarp();
    };
    // dV += P_t^T dO_t (KV only): needs P_t alone
    auto issue_dv = [&](int b, int slot, bool first) {
      const uint64_t so = static_cast<uint64_t>(slot * C::STAGE_BYTES) >> 4;
      const uint64_t w0 = dWm + so;
      const uint32_t a0 = tmem + col_buf(b);
      if (ptx::elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kStr / 16; ++kk) {
          const uint64_t bo = static_cast<uint64_t>(kk * 16 * 128) >> 4;  // 16 streamed rows
          const uint32_t acc = (kk > 0 || !first) ? 1u : 0u;
          // streamed rows 16kk..16kk+15: half kk/2, 16-bit pairs from column 8*(kk%2)
          const uint32_t a_col = a0 + (kk >> 1) * 32 + (kk & 1) * 8;
          ptx::mma_f16_ts(tmem + kColAcc1, a_col, w0 + bo, idG, acc);
        }
      }
      __syncwarp();
    };
    // dK += dS_t^T Q_t (KV) or dQ += dS_t K_t (Q); frees the stage
    auto issue_ds = [&](int b, int slot, bool first) {
      const uint64_t so = static_cast<uint64_t>(slot * C::STAGE_BYTES) >> 4;
      const uint64_t u0 = dUm + so;
      const uint32_t a0 = tmem + col_buf(b);
      if (ptx::elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kStr / 16; ++kk) {
          const uint64_t bo = static_cast<uint64_t>(kk * 16 * 128) >> 4;
          const uint32_t acc = (kk > 0 || !first) ? 1u : 0u;
          const uint32_t a_col = a0 + (kk >> 1) * 32 + (kk & 1) * 8;
          ptx::mma_f16_ts(tmem + C::COL_ACC2, a_col + 64, u0 + bo, idG, acc);
        }
        ptx::mma_commit(&stage_empty[slot]);
      }
      __syncwarp();
    };
    // every lane waits; the result is made warp-uniform
    auto wait = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      const bool good = ptx::mbar_wait(bar, parity, status, status_word(kKern, site));
      return __all_sync(0xffffffffu, good);
    };

    bool ok = C::XY_TMEM ? wait(res_tmem, 0, kSiteMmaRes) : wait(res_full, 0, kSiteMmaRes);
    if (ok) ok = wait(&stage_full[0], 0, kSiteMmaStage);
    if (ok) {
      ptx::tc_fence_after();
      issue_scores(0, 0);
    }
    for (int it = 0; ok && it < n; ++it) {
      const int b = it & 1;
      if (it + 1 < n) {
        // scores of the next tile into the other buffer: its previous
        // contents (tile it-1) were read by tile it-1's gradient products,
        // issued earlier by the same lane and so executed earlier
        const int s1 = (it + 1) % ST;
        ok = wait(&stage_full[s1], ((it + 1) / ST) & 1, kSiteMmaStage);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_scores(b ^ 1, s1);
      }
      if constexpr (KV) {
        ok = wait(&p_half[b], (it >> 1) & 1, kSiteMmaP);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_dv(b, it % ST, it == 0);
      }
      ok = wait(&p_full[b], (it >> 1) & 1, kSiteMmaP);
      if (!ok) break;
      ptx::tc_fence_after();
      issue_ds(b, it % ST, it == 0);
    }
    // every MMA issued must be complete before TMEM is freed
    if (ptx::elect_one_sync()) {
      if (ok) ptx::mma_commit(acc_full);
      ptx::mma_commit(mma_done);
    }
    __syncwarp();
    mbar_drain(mma_done, 0);
  } else {
    // ---------------------------------------------------------------- elementwise
    const int quarter = warp & 3;                      // TMEM lanes 32*quarter..
    const int half = warp >> 2;                        // columns 32*half.. of each tile
    const int row = quarter * 32 + lane;               // TMEM lane = resident row
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t t_half = t_lane + static_cast<uint32_t>(half * 32);
    const int rrow = w.r0 + row;                       // KV: key index; Q: query row
    float l2_row = 0.f, dd_row = 0.f;
    if constexpr (!KV) {
      const size_t ro = static_cast<size_t>(w.res_bh) * Tq_pad + rrow;  // rrow < Tq_pad
      l2_row = ws_l2[ro];
      dd_row = ws_dd[ro];
    }
    const float2 sl2 = make_float2(scale_log2, scale_log2);
    bool ok = true;
    if constexpr (C::XY_TMEM) {
      // row `row` of X (warps 0-3) or Y (warps 4-7), from the 128-byte
      // swizzled tile (16-byte chunk c of a row r sits at chunk c ^ (r % 8)),
      // into D/2 columns of TMEM as 16-bit pairs in K order: the A-operand
      // layout of the score products
      ok = ptx::mbar_wait(res_full, 0, status, status_word(kKern, kSiteEltRes));
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        const uint8_t* tile = smem + (half ? C::OFF_Y : C::OFF_X);
#pragma unroll
        for (int c32 = 0; c32 < D / 64; ++c32) {   // 32 columns = one 64-element sub-tile
          uint32_t words[32];
          const uint8_t* sub = tile + c32 * kSubRes + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(sub + ((c ^ (row & 7)) << 4));
            words[4 * c] = v.x;
            words[4 * c + 1] = v.y;
            words[4 * c + 2] = v.z;
            words[4 * c + 3] = v.w;
          }
          ptx::tmem_st_32x32b_x32(t_lane + (half ? C::COL_Y : C::COL_X) + c32 * 32, words);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(res_tmem);
      }
    }
    for (int it = 0; ok && it < n; ++it) {
      const int b = it & 1;
      const int slot = it % ST;
      ok = ptx::mbar_wait(&sp_full[b], (it >> 1) & 1, status, status_word(kKern, kSiteEltS));
      if constexpr (KV) {
        // the row vectors arrived with the tile (TMA writes are visible to
        // the threads that observe the stage barrier)
        if (ok)
          ok = ptx::mbar_wait(&stage_full[slot], (it / ST) & 1, status,
                              status_word(kKern, kSiteEltStage));
      }
      // tcgen05.ld/st/wait are warp-collective: the whole warp takes every
      // branch around them
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      int sbh, s0;
      bwd_item(w, it, &sbh, &s0);
      s0 += half * 32;  // streamed row of this warp's column 0
      if constexpr (KV) {
        // The 16-lane shape: each thread holds four keys (lanes i/4 + {0, 8,
        // 16, 24} of the quarter) at eight of the warp's 32 columns (8r + c2
        // and the next, r = 0..3), so it needs only those columns' lse and D
        // (8-byte loads that four lanes share).
        const float* v0 = reinterpret_cast<const float*>(smem + C::OFF_RING +
                                                         slot * C::STAGE_BYTES + 2 * C::STR_BYTES) +
                          half * 32;
        const int c2 = 2 * (lane & 3);
        float2 nl[4], nd[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float2 l = *reinterpret_cast<const float2*>(v0 + 8 * r + c2);
          const float2 d2 = *reinterpret_cast<const float2*>(v0 + kStr + 8 * r + c2);
          nl[r] = make_float2(-l.x, -l.y);
          nd[r] = make_float2(-d2.x, -d2.y);
        }
        // query s0 + c sees key x iff c >= cmin[x]
        int cmin[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int kx = w.r0 + quarter * 32 + 16 * (x >> 1) + (lane >> 2) + 8 * (x & 1);
          cmin[x] = causal ? kx - off - s0 : INT_MIN / 2;
          if (kx >= T_kv) cmin[x] = 32;  // key past the end: nothing visible
        }
        const bool all_visible =
            __all_sync(0xffffffffu, max(max(cmin[0], cmin[1]), max(cmin[2], cmin[3])) <= 0);
        // sr[16h + 4r + 2e + j] = S(key (h, e), column 8r + c2 + j); dP at +32
        const uint32_t col = col_buf(b) + half * 32;
        uint32_t sr[64];
        ptx::tmem_ld_16x256b_x4(t_lane + col, *reinterpret_cast<uint32_t(*)[16]>(&sr[0]));
        ptx::tmem_ld_16x256b_x4(t_lane + (16u << 16) + col, *reinterpret_cast<uint32_t(*)[16]>(&sr[16]));
        ptx::tmem_ld_16x256b_x4(t_lane + col + 64, *reinterpret_cast<uint32_t(*)[16]>(&sr[32]));
        ptx::tmem_ld_16x256b_x4(t_lane + (16u << 16) + col + 64,
                                *reinterpret_cast<uint32_t(*)[16]>(&sr[48]));
        tmem_wait_ld_64(sr);
        const float* s = reinterpret_cast<const float*>(sr);
        const float* dp = reinterpret_cast<const float*>(sr + 32);
        float2 pp[16];  // pp[8h + 2r + e]
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 16 * h2 + 4 * r + 2 * e;
              const float2 x = __ffma2_rn(make_float2(s[i], s[i + 1]), sl2, nl[r]);
              pp[8 * h2 + 2 * r + e] = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
            }
        if (!all_visible) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int c = 8 * r + c2, m = cmin[2 * h2 + e];
                float2& v = pp[8 * h2 + 2 * r + e];
                v.x = c >= m ? v.x : 0.f;
                v.y = c + 1 >= m ? v.y : 0.f;
              }
        }
        // P over the first 16 columns of this warp's half of S (the pair of
        // columns 8r + c2 is word 4r + lane%4), released at once: dV += P^T dO
        // runs while dS is formed
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) pk[j] = pack2<BF16>(pp[8 * h2 + j].x, pp[8 * h2 + j].y);
          ptx::tmem_st_16x128b_x4(t_lane + (static_cast<uint32_t>(16 * h2) << 16) + col, pk);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&p_half[b]);
        // dS over the first 16 columns of this warp's half of dP
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t gk[8];
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 16 * h2 + 4 * r + 2 * e;
              const float2 g = __fmul2_rn(pp[8 * h2 + 2 * r + e],
                                          __fadd2_rn(make_float2(dp[i], dp[i + 1]), nd[r]));
              gk[2 * r + e] = pack2<BF16>(g.x, g.y);
            }
          ptx::tmem_st_16x128b_x4(t_lane + (static_cast<uint32_t>(16 * h2) << 16) + col + 64, gk);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&p_full[b]);
      } else {
        uint32_t sr[64];
        ptx::tmem_ld_32x32b_x32(t_half + col_buf(b), *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        ptx::tmem_ld_32x32b_x32(t_half + col_buf(b) + 64,
                                *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_ld_64(sr);
        const float* s = reinterpret_cast<const float*>(sr);        // scores, 32 columns
        const float* dp = reinterpret_cast<const float*>(sr + 32);  // dP, same columns
        const float2 nl = make_float2(-l2_row, -l2_row);
        const float2 nd = make_float2(-dd_row, -dd_row);
        // columns [0, cmax] of this row are visible
        const int cmax = (causal ? min(rrow + off, T_kv - 1) : T_kv - 1) - s0;
        const bool all_visible = __all_sync(0xffffffffu, cmax >= 31);
        float2 pp[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 x = __ffma2_rn(make_float2(s[2 * j], s[2 * j + 1]), sl2, nl);
          pp[j] = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
        }
        if (!all_visible) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            pp[c >> 1].x = c <= cmax ? pp[c >> 1].x : 0.f;
            pp[c >> 1].y = c + 1 <= cmax ? pp[c >> 1].y : 0.f;
          }
        }
        uint32_t gk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 g = __fmul2_rn(pp[j], __fadd2_rn(make_float2(dp[2 * j], dp[2 * j + 1]), nd));
          gk[j] = pack2<BF16>(g.x, g.y);
        }
        // dS over the first 16 columns of this warp's half of dP
        ptx::tmem_st_32x32b_x16(t_half + col_buf(b) + 64, gk);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&p_full[b]);
      }
    }
    if (ok) {
      // -------------------------------------------------------------- epilogue
      ok = ptx::mbar_wait(acc_full, 0, status, status_word(kKern, kSiteEltAcc));
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        ptx::tc_fence_after();
        const int T_out = KV ? T_kv : T_q;
        const bool write = rrow < T_out;
        constexpr int HALF_D = D / 2;  // output columns of this warp
#pragma unroll
        for (int a = KV ? 0 : 1; a < 2; ++a) {
          uint8_t* dst = reinterpret_cast<uint8_t*>(a == 0 ? out1 : out2) +
                         (static_cast<size_t>(w.res_bh) * T_out + (write ? rrow : 0)) * D * 2 +
                         half * HALF_D * 2;
          const float mul = a == 0 ? 1.f : scale;
          const uint32_t col = (a == 0 ? kColAcc1 : C::COL_ACC2) + half * HALF_D;
#pragma unroll
          for (int c = 0; c < HALF_D / 32; ++c) {
            uint32_t raw[32];
            ptx::tmem_ld_32x32b_x32(t_lane + col + c * 32, raw);
            tmem_wait_ld_32(raw);
            if (write) {
#pragma unroll
              for (int g8 = 0; g8 < 4; ++g8) {
                const float* f = reinterpret_cast<const float*>(&raw[g8 * 8]);
                uint4 v;
                v.x = pack2<BF16>(f[0] * mul, f[1] * mul);
                v.y = pack2<BF16>(f[2] * mul, f[3] * mul);
                v.z = pack2<BF16>(f[4] * mul, f[5] * mul);
                v.w = pack2<BF16>(f[6] * mul, f[7] * mul);
                *reinterpret_cast<uint4*>(dst + (c * 32 + g8 * 8) * 2) = v;
              }
            }
          }
        }
      }
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// dK/dV at d = 64 with 128-row streamed query tiles. One CTA per (key/value
// head, 128-key tile): K and V stay in shared memory and the CTA streams
// 128-row tiles of Q and dO (with their lse*log2(e) and D) through a 5-stage
// ring, for every query head of the group and, causally, only tiles with a
// row that sees the key tile. The keys sit on the TMEM lanes. Per tile t the
// tensor core computes
//   S_t^T = K Q_t^T and dP_t^T = V dO_t^T   (M = 128 keys, N = 128 queries, K = 64)
// from shared memory into TMEM (S in two buffers, dP in one). Elementwise
// warp w owns the keys 32*(w%4).. (its TMEM lane quarter) and the 64 queries
// 64*(w/4).. of each tile. It reads them with the 16-lane shape: each thread
// holds four keys (lanes i/4 + {0, 8, 16, 24}) at 16 of the columns (two of
// every eight), so it needs only those 16 columns' lse and D from the stage
// (8-byte loads that four lanes share) rather than all 64 in every lane. It
// forms P = 2^(scale*log2e*S - lse*log2e) and stores it as 16-bit pairs over
// the first 32 of its 64 S columns (16x128b shape: the pair of columns
// 8r + 2(i%4) is word 4r + i%4 of the lane); once dP is there it forms
// dS = P * (dP - D) and stores it the same way over its dP columns. The
// tensor core accumulates dV += P_t^T dO_t and dK += dS_t^T Q_t (M = 128
// keys, N = 64, K = 128 queries) with A read from TMEM and B the streamed
// tile read MN-major, so shared memory carries only the four products' B
// operands and the score products' A. Issue order dV(t), dK(t), dP(t+1),
// S(t+2): every product overwrites a buffer only after the products that
// read it (one thread's MMAs execute in order), and the warps form P(t+1)
// while dK(t) and dP(t+1) run, dS(t+1) while dV(t+1) and S(t+2) run. P's
// barrier alternates between two, so that none can complete a second phase
// before the issuer has waited for the first: P(t+2) needs S(t+2), issued
// only after the wait for P(t).
// TMEM: S [0,256), dP [256,384), dV [384,448), dK [448,512).
// ---------------------------------------------------------------------------
namespace kv128 {
constexpr int kRows = 128;                      // keys per CTA; queries per streamed tile
constexpr int kTile = kRows * 64 * 2;           // one [128 rows][64] 16-bit tile (128-byte rows)
constexpr int kStages = 5;
constexpr int kStageBytes = 2 * kTile + 1024;   // Q, dO, then lse*log2e [128] and D [128]
constexpr int OFF_K = 0;
constexpr int OFF_V = kTile;
constexpr int OFF_RING = 2 * kTile;
constexpr int OFF_BAR = OFF_RING + kStages * kStageBytes;
// res_full, stage_full[5], stage_empty[5], s_full[2], dp_full, p_ready[2], ds_ready, acc_full,
// mma_done
constexpr int N_BARS = 1 + 2 * kStages + 2 + 6;
constexpr int OFF_TMEMPTR = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
constexpr uint32_t COL_S = 0, COL_DP = 256, COL_DV = 384, COL_DK = 448;
static_assert(kStageBytes % 1024 == 0 && OFF_RING % 1024 == 0, "atoms");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

// Unit u (heaviest first under a causal mask: key tile 0 sees every query):
// the key/value head and 128-key tile, and the streamed 128-row query tiles.
struct Unit {
  int res_bh, r0, str_bh0, t_first, per_head, n;
};
__device__ __forceinline__ Unit unit_of(int u, int BH_kv, int T_q, int T_kv, int causal, int h,
                                        int h_kv) {
  const int group = h / h_kv;
  const int off = T_kv - T_q;
  Unit w;
  w.res_bh = u % BH_kv;
  w.r0 = (u / BH_kv) * kRows;
  const int b = w.res_bh / h_kv, kvh = w.res_bh % h_kv;
  w.str_bh0 = b * h + kvh * group;
  const int first_row = causal ? max(0, w.r0 - off) : 0;  // key r0 is seen by rows >= r0 - off
  w.t_first = first_row / kRows;
  w.per_head = (T_q + kRows - 1) / kRows - w.t_first;
  w.n = max(0, w.per_head) * group;
  return w;
}
__device__ __forceinline__ void item_of(const Unit& w, int it, int* bh, int* s0) {
  const int g = it / w.per_head;
  *bh = w.str_bh0 + g;
  *s0 = (w.t_first + (it - g * w.per_head)) * kRows;
}
}  // namespace kv128

template <bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kv128_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                     const float* __restrict__ ws_l2, const float* __restrict__ ws_dd, int Tq_pad,
                     void* __restrict__ dv_out, void* __restrict__ dk_out, int T_q, int T_kv,
                     int BH_kv, int h, int h_kv, float scale, float scale_log2, int causal,
                     unsigned int* __restrict__ status) {
  using namespace kv128;
  constexpr int ST = kStages;
  constexpr uint32_t kKern = kKernBwdKV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* res_full = bars;
  uint64_t* stage_full = bars + 1;
  uint64_t* stage_empty = stage_full + ST;
  uint64_t* s_full = stage_empty + ST;
  uint64_t* dp_full = s_full + 2;
  uint64_t* p_ready = dp_full + 1;  // [2]
  uint64_t* ds_ready = p_ready + 2;
  uint64_t* acc_full = ds_ready + 1;
  uint64_t* mma_done = acc_full + 1;
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + OFF_TMEMPTR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Unit w = unit_of(static_cast<int>(blockIdx.x), BH_kv, T_q, T_kv, causal, h, h_kv);
  const int n = w.n;
  const int off = T_kv - T_q;

  if (threadIdx.x == 0) {
    ptx::mbar_init(res_full, 1);
    for (int i = 0; i < ST; ++i) {
      ptx::mbar_init(&stage_full[i], 1);
      ptx::mbar_init(&stage_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(&s_full[b], 1);
    ptx::mbar_init(dp_full, 1);
    for (int b = 0; b < 2; ++b) ptx::mbar_init(&p_ready[b], kEltThreads);
    ptx::mbar_init(ds_ready, kEltThreads);
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(mma_done, 1);
    ptx::fence_mbarrier_init();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(tmem_ptr, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  if (warp == kWarpProd) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmK);
      ptx::prefetch_tensormap(&tmV);
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmO);
      const uint64_t pol_str = ptx::policy_evict_last();
      const uint64_t pol_res = ptx::policy_evict_first();
      ptx::mbar_arrive_expect_tx(res_full, 2 * kTile);
      ptx::tma_load_3d(smem + OFF_K, &tmK, res_full, 0, w.r0, w.res_bh, pol_res);
      ptx::tma_load_3d(smem + OFF_V, &tmV, res_full, 0, w.r0, w.res_bh, pol_res);
      bool ok = true;
      int it = 0;
      for (; it < n; ++it) {
        const int slot = it % ST;
        ok = ptx::mbar_wait(&stage_empty[slot], ((it / ST) & 1) ^ 1, status,
                            status_word(kKern, kSiteProdStage));
        if (!ok) break;
        int sbh, s0;
        item_of(w, it, &sbh, &s0);
        uint8_t* stg = smem + OFF_RING + slot * kStageBytes;
        ptx::mbar_arrive_expect_tx(&stage_full[slot], 2 * kTile + 2 * kRows * 4);
        ptx::tma_load_3d(stg, &tmQ, &stage_full[slot], 0, s0, sbh, pol_str);
        ptx::tma_load_3d(stg + kTile, &tmO, &stage_full[slot], 0, s0, sbh, pol_str);
        const size_t vo = static_cast<size_t>(sbh) * Tq_pad + s0;
        ptx::bulk_load(stg + 2 * kTile, ws_l2 + vo, kRows * 4, &stage_full[slot]);
        ptx::bulk_load(stg + 2 * kTile + kRows * 4, ws_dd + vo, kRows * 4, &stage_full[slot]);
      }
      if (!ok) {
        // let the copies in flight land before the CTA's shared memory goes
        mbar_drain(res_full, 0);
        for (int i = (it > ST ? it - ST : 0); i < it; ++i) mbar_drain(&stage_full[i % ST], (i / ST) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = ptx::make_idesc_f16(BF16, kRows, kRows, false, false);
    constexpr uint32_t idG = ptx::make_idesc_f16(BF16, kRows, 64, false, true);
    const uint32_t sR = ptx::smem_u32(smem + OFF_RING);
    const uint64_t dK = ptx::make_sdesc_sw128(ptx::smem_u32(smem + OFF_K), 16, 1024);
    const uint64_t dV = ptx::make_sdesc_sw128(ptx::smem_u32(smem + OFF_V), 16, 1024);
    auto stage_desc = [&](int slot, int which, bool mn) {
      return ptx::make_sdesc_sw128(sR + slot * kStageBytes + which * kTile, mn ? kTile : 16, 1024);
    };
    // S^T (which = 0: K against Q) or dP^T (which = 1: V against dO)
    auto issue_score = [&](int which, uint32_t d_col, int slot, uint64_t* bar) {
      const uint64_t a0 = which == 0 ? dK : dV;
      const uint64_t b0 = stage_desc(slot, which, false);
      if (ptx::elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f16_ss(tmem + d_col, a0 + kk * 2, b0 + kk * 2, idS, kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar);
      }
      __syncwarp();
    };
    // dV += P^T dO (a_col = the P buffer) or dK += dS^T Q (a_col = dP's)
    auto issue_grad = [&](uint32_t acc_col, uint32_t a_col, int slot, int which, bool first) {
      const uint64_t b0 = stage_desc(slot, which, true);
      if (ptx::elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk) {
          // queries 16kk..16kk+15: warp half kk/4, 16-bit pairs from column 8*(kk%4)
          const uint32_t a = tmem + a_col + (kk >> 2) * 64 + (kk & 3) * 8;
          const uint64_t step = static_cast<uint64_t>(kk * 16 * 128) >> 4;  // 16 query rows
          ptx::mma_f16_ts(tmem + acc_col, a, b0 + step, idG, (kk > 0 || !first) ? 1u : 0u);
        }
      }
      __syncwarp();
    };
    auto wait = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      const bool good = ptx::mbar_wait(bar, parity, status, status_word(kKern, site));
      return __all_sync(0xffffffffu, good);
    };

    bool ok = wait(res_full, 0, kSiteMmaRes);
    for (int i = 0; ok && i < 2 && i < n; ++i) {
      ok = wait(&stage_full[i], 0, kSiteMmaStage);
      if (!ok) break;
      ptx::tc_fence_after();
      issue_score(0, COL_S + i * 128, i, &s_full[i]);
      if (i == 0) issue_score(1, COL_DP, 0, dp_full);
    }
    for (int it = 0; ok && it < n; ++it) {
      const int b = it & 1;
      const int slot = it % ST;
      ok = wait(&p_ready[b], (it >> 1) & 1, kSiteMmaP);
      if (!ok) break;
      ptx::tc_fence_after();
      issue_grad(COL_DV, COL_S + b * 128, slot, 1, it == 0);
      ok = wait(ds_ready, it & 1, kSiteMmaP);
      if (!ok) break;
      ptx::tc_fence_after();
      issue_grad(COL_DK, COL_DP, slot, 0, it == 0);
      if (ptx::elect_one_sync()) ptx::mma_commit(&stage_empty[slot]);
      __syncwarp();
      // the next tile's stage was waited for with its scores
      if (it + 1 < n) issue_score(1, COL_DP, (it + 1) % ST, dp_full);
      if (it + 2 < n) {
        const int s2 = (it + 2) % ST;
        ok = wait(&stage_full[s2], ((it + 2) / ST) & 1, kSiteMmaStage);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_score(0, COL_S + b * 128, s2, &s_full[b]);
      }
    }
    // every MMA issued must be complete before TMEM is freed
    if (ptx::elect_one_sync()) {
      if (ok) ptx::mma_commit(acc_full);
      ptx::mma_commit(mma_done);
    }
    __syncwarp();
    mbar_drain(mma_done, 0);
  } else {
    // ---------------------------------------------------------------- elementwise
    const int quarter = warp & 3;                    // TMEM lanes 32*quarter..
    const int half = warp >> 2;                      // queries 64*half.. of each tile
    const int key = w.r0 + quarter * 32 + lane;      // the epilogue's key (32x32b shape)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float2 sl2 = make_float2(scale_log2, scale_log2);
    bool ok = true;
    for (int it = 0; ok && it < n; ++it) {
      const int b = it & 1;
      const int slot = it % ST;
      ok = ptx::mbar_wait(&s_full[b], (it >> 1) & 1, status, status_word(kKern, kSiteEltS));
      // the row vectors arrived with the tile (TMA writes are visible to the
      // threads that observe the stage barrier)
      if (ok)
        ok = ptx::mbar_wait(&stage_full[slot], (it / ST) & 1, status,
                            status_word(kKern, kSiteEltStage));
      // tcgen05.ld/st/wait are warp-collective: the whole warp takes every
      // branch around them
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      int sbh, s0;
      item_of(w, it, &sbh, &s0);
      // lse*log2e and D of this thread's 16 query columns: 8r + c2 and the
      // next, r = 0..7 (4 distinct 8-byte words per warp load)
      const float* lvec = reinterpret_cast<const float*>(smem + OFF_RING + slot * kStageBytes +
                                                         2 * kTile) + half * 64;
      const float* dvec = lvec + kRows;
      const int c2 = 2 * (lane & 3);
      // this thread's four keys: rows 16h + lane/4 + 8e of the warp's quarter
      // (h, e in {0, 1}); query s0 + 64*half + c sees key x iff c >= cmin[x]
      int cmin[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int kx = w.r0 + quarter * 32 + 16 * (x >> 1) + (lane >> 2) + 8 * (x & 1);
        cmin[x] = causal ? kx - off - (s0 + half * 64) : INT_MIN / 2;
        if (kx >= T_kv) cmin[x] = 64;  // key past the end: nothing visible
      }
      const bool all_visible =
          __all_sync(0xffffffffu, max(max(cmin[0], cmin[1]), max(cmin[2], cmin[3])) <= 0);
      const uint32_t col_s = COL_S + b * 128 + half * 64;
      const uint32_t col_dp = COL_DP + half * 64;
      float2 nl[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float2 l = *reinterpret_cast<const float2*>(lvec + 8 * r + c2);
        nl[r] = make_float2(-l.x, -l.y);
      }
      // S of lanes 0-15 (sr[0..31]) and 16-31 (sr[32..63]) of the quarter:
      // sr[32h + 4r + 2e + j] = S(key (h, e), column 8r + c2 + j)
      uint32_t sr[64];
      ptx::tmem_ld_16x256b_x8(t_lane + col_s, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      ptx::tmem_ld_16x256b_x8(t_lane + (16u << 16) + col_s, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld_64(sr);
      const float* s = reinterpret_cast<const float*>(sr);
      // pp[16h + 2r + e]: key (h, e), columns 8r + c2 and 8r + c2 + 1
      float2 pp[32];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 32 * h2 + 4 * r + 2 * e;
            const float2 x = __ffma2_rn(make_float2(s[i], s[i + 1]), sl2, nl[r]);
            pp[16 * h2 + 2 * r + e] = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
          }
      if (!all_visible) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = 8 * r + c2, m = cmin[2 * h2 + e];
              float2& v = pp[16 * h2 + 2 * r + e];
              v.x = c >= m ? v.x : 0.f;
              v.y = c + 1 >= m ? v.y : 0.f;
            }
      }
      // P as 16-bit pairs over the first 32 of the warp's 64 S columns: the
      // pair of columns 8r + c2 is word 4r + lane%4, which the 16x128b shape
      // takes from register 2r (lane lane/4) and 2r + 1 (lane lane/4 + 8)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack2<BF16>(pp[16 * h2 + j].x, pp[16 * h2 + j].y);
        ptx::tmem_st_16x128b_x8(t_lane + (static_cast<uint32_t>(16 * h2) << 16) + col_s, pk);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&p_ready[b]);

      ok = ptx::mbar_wait(dp_full, it & 1, status, status_word(kKern, kSiteEltS));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      float2 nd[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float2 d2 = *reinterpret_cast<const float2*>(dvec + 8 * r + c2);
        nd[r] = make_float2(-d2.x, -d2.y);
      }
      uint32_t dr[64];
      ptx::tmem_ld_16x256b_x8(t_lane + col_dp, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      ptx::tmem_ld_16x256b_x8(t_lane + (16u << 16) + col_dp, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tmem_wait_ld_64(dr);
      const float* dp = reinterpret_cast<const float*>(dr);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t gk[16];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 32 * h2 + 4 * r + 2 * e;
            const float2 g = __fmul2_rn(pp[16 * h2 + 2 * r + e],
                                        __fadd2_rn(make_float2(dp[i], dp[i + 1]), nd[r]));
            gk[2 * r + e] = pack2<BF16>(g.x, g.y);
          }
        ptx::tmem_st_16x128b_x8(t_lane + (static_cast<uint32_t>(16 * h2) << 16) + col_dp, gk);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ds_ready);
    }
    if (ok) {
      // -------------------------------------------------------------- epilogue
      ok = ptx::mbar_wait(acc_full, 0, status, status_word(kKern, kSiteEltAcc));
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        ptx::tc_fence_after();
        const bool write = key < T_kv;  // accumulator lanes are keys
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          uint8_t* dst = reinterpret_cast<uint8_t*>(a == 0 ? dv_out : dk_out) +
                         (static_cast<size_t>(w.res_bh) * T_kv + (write ? key : 0)) * 64 * 2 +
                         half * 32 * 2;
          const float mul = a == 0 ? 1.f : scale;
          uint32_t raw[32];
          ptx::tmem_ld_32x32b_x32(t_lane + (a == 0 ? COL_DV : COL_DK) + half * 32, raw);
          tmem_wait_ld_32(raw);
          if (write) {
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              const float* f = reinterpret_cast<const float*>(&raw[g8 * 8]);
              uint4 v;
              v.x = pack2<BF16>(f[0] * mul, f[1] * mul);
              v.y = pack2<BF16>(f[2] * mul, f[3] * mul);
              v.z = pack2<BF16>(f[4] * mul, f[5] * mul);
              v.w = pack2<BF16>(f[6] * mul, f[7] * mul);
              *reinterpret_cast<uint4*>(dst + g8 * 16) = v;
            }
          }
        }
      }
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dQ at d = 64 with 128-key streamed tiles. One CTA per (query head, 128-row
// query tile), heaviest first: Q and dO stay (copied once into TMEM as the A
// operands of the score products) and the CTA streams 128-key tiles of K and
// V through a 5-stage ring, causally up to the diagonal. The query rows sit on
// the TMEM lanes; per key tile t the tensor core computes
//   S_t = Q K_t^T and dP_t = dO V_t^T   (M = 128 rows, N = 128 keys, K = 64)
// with A from TMEM and B from shared memory, S into one buffer and dP into
// one of two. Elementwise thread (warp w, lane i) owns row 32*(w%4)+i (its
// lse and D are two registers) and the 64 keys 64*(w/4).. of each tile: it
// loads its S values and releases the S buffer at once, forms P, waits for
// dP, forms dS = P * (dP - D) and stores it as 16-bit pairs over the first
// 32 of its 64 dP columns; the tensor core accumulates dQ += dS_t K_t (M =
// 128 rows, N = 64, K = 128 keys; A from TMEM, B the K tile read MN-major).
// Issue order per tile: S(t+1) once S(t) is loaded, then dQ(t) once dS(t) is
// stored, then dP(t+2) into the buffer dQ(t) has just read (one thread's
// MMAs execute in order), so the scores of a tile are ready before the warps
// reach it. TMEM: S [0,128), dP [128,384), dQ [384,448), Q [448,480),
// dO [480,512).
// ---------------------------------------------------------------------------
namespace q128 {
constexpr int kRows = 128;                // query rows per CTA; keys per streamed tile
constexpr int kTile = kRows * 64 * 2;     // one [128 rows][64] 16-bit tile (128-byte rows)
constexpr int kStages = 5;
constexpr int kStageBytes = 2 * kTile;    // K, V
constexpr int OFF_Q = 0;
constexpr int OFF_DO = kTile;
constexpr int OFF_RING = 2 * kTile;
constexpr int OFF_BAR = OFF_RING + kStages * kStageBytes;
// res_full, res_tmem, stage_full[5], stage_empty[5], s_full, s_free, dp_full[2], ds_ready[2],
// acc_full, mma_done
constexpr int N_BARS = 2 + 2 * kStages + 2 + 4 + 2;
constexpr int OFF_TMEMPTR = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 384, COL_Q = 448, COL_DO = 480;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
}  // namespace q128

template <bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_q128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const float* __restrict__ ws_l2, const float* __restrict__ ws_dd, int Tq_pad,
                    void* __restrict__ dq_out, int T_q, int T_kv, int BH, int n_qt, int h, int h_kv,
                    float scale, float scale_log2, int causal, unsigned int* __restrict__ status) {
  using namespace q128;
  constexpr int ST = kStages;
  constexpr uint32_t kKern = kKernBwdQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* res_full = bars;
  uint64_t* res_tmem = bars + 1;
  uint64_t* stage_full = bars + 2;
  uint64_t* stage_empty = stage_full + ST;
  uint64_t* s_full = stage_empty + ST;
  uint64_t* s_free = s_full + 1;
  uint64_t* dp_full = s_free + 1;   // [2]
  uint64_t* ds_ready = dp_full + 2;  // [2]
  uint64_t* acc_full = ds_ready + 2;
  uint64_t* mma_done = acc_full + 1;
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + OFF_TMEMPTR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = h / h_kv;
  const int off = T_kv - T_q;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int r0 = (n_qt - 1 - static_cast<int>(blockIdx.x) / BH) * kRows;
  const int kv_bh = bh / group;  // (b * h + i) / group = b * h_kv + i / group
  const int last_row = min(T_q, r0 + kRows) - 1;
  const int last_key = causal ? min(T_kv - 1, last_row + off) : T_kv - 1;  // >= 0: T_q <= T_kv
  const int n = last_key / kRows + 1;

  if (threadIdx.x == 0) {
    ptx::mbar_init(res_full, 1);
    ptx::mbar_init(res_tmem, kEltThreads);
    for (int i = 0; i < ST; ++i) {
      ptx::mbar_init(&stage_full[i], 1);
      ptx::mbar_init(&stage_empty[i], 1);
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(s_free, kEltThreads);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&dp_full[b], 1);
      ptx::mbar_init(&ds_ready[b], kEltThreads);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(mma_done, 1);
    ptx::fence_mbarrier_init();
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(tmem_ptr, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  if (warp == kWarpProd) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmO);
      ptx::prefetch_tensormap(&tmK);
      ptx::prefetch_tensormap(&tmV);
      // the streamed tiles are read by every query tile of the head: keep
      // them in L2; the resident ones once
      const uint64_t pol_str = ptx::policy_evict_last();
      const uint64_t pol_res = ptx::policy_evict_first();
      ptx::mbar_arrive_expect_tx(res_full, 2 * kTile);
      ptx::tma_load_3d(smem + OFF_Q, &tmQ, res_full, 0, r0, bh, pol_res);
      ptx::tma_load_3d(smem + OFF_DO, &tmO, res_full, 0, r0, bh, pol_res);
      bool ok = true;
      int it = 0;
      for (; it < n; ++it) {
        const int slot = it % ST;
        ok = ptx::mbar_wait(&stage_empty[slot], ((it / ST) & 1) ^ 1, status,
                            status_word(kKern, kSiteProdStage));
        if (!ok) break;
        uint8_t* stg = smem + OFF_RING + slot * kStageBytes;
        ptx::mbar_arrive_expect_tx(&stage_full[slot], 2 * kTile);
        ptx::tma_load_3d(stg, &tmK, &stage_full[slot], 0, it * kRows, kv_bh, pol_str);
        ptx::tma_load_3d(stg + kTile, &tmV, &stage_full[slot], 0, it * kRows, kv_bh, pol_str);
      }
      if (!ok) {
        // let the copies in flight land before the CTA's shared memory goes
        mbar_drain(res_full, 0);
        for (int i = (it > ST ? it - ST : 0); i < it; ++i) mbar_drain(&stage_full[i % ST], (i / ST) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = ptx::make_idesc_f16(BF16, kRows, kRows, false, false);
    constexpr uint32_t idG = ptx::make_idesc_f16(BF16, kRows, 64, false, true);
    const uint32_t sR = ptx::smem_u32(smem + OFF_RING);
    auto stage_desc = [&](int slot, int which, bool mn) {
      return ptx::make_sdesc_sw128(sR + slot * kStageBytes + which * kTile, mn ? kTile : 16, 1024);
    };
    // S (which = 0: Q against K) or dP (which = 1: dO against V)
    auto issue_score = [&](int which, uint32_t d_col, int slot, uint64_t* bar) {
      const uint32_t a0 = tmem + (which == 0 ? COL_Q : COL_DO);
      const uint64_t b0 = stage_desc(slot, which, false);
      if (ptx::elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f16_ts(tmem + d_col, a0 + kk * 8, b0 + kk * 2, idS, kk > 0 ? 1u : 0u);
        ptx::mma_commit(bar);
      }
      __syncwarp();
    };
    // dQ += dS K, dS over the first 32 columns of each half of dP buffer b
    auto issue_dq = [&](int b, int slot, bool first) {
      const uint64_t b0 = stage_desc(slot, 0, true);
      if (ptx::elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk) {
          // keys 16kk..16kk+15: warp half kk/4, 16-bit pairs from column 8*(kk%4)
          const uint32_t a = tmem + COL_DP + b * 128 + (kk >> 2) * 64 + (kk & 3) * 8;
          const uint64_t step = static_cast<uint64_t>(kk * 16 * 128) >> 4;  // 16 key rows
          ptx::mma_f16_ts(tmem + COL_DQ, a, b0 + step, idG, (kk > 0 || !first) ? 1u : 0u);
        }
        ptx::mma_commit(&stage_empty[slot]);
      }
      __syncwarp();
    };
    auto wait = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
      const bool good = ptx::mbar_wait(bar, parity, status, status_word(kKern, site));
      return __all_sync(0xffffffffu, good);
    };

    bool ok = wait(res_tmem, 0, kSiteMmaRes);
    for (int i = 0; ok && i < 2 && i < n; ++i) {
      ok = wait(&stage_full[i], 0, kSiteMmaStage);
      if (!ok) break;
      ptx::tc_fence_after();
      if (i == 0) issue_score(0, COL_S, 0, s_full);
      issue_score(1, COL_DP + i * 128, i, &dp_full[i]);
    }
    for (int it = 0; ok && it < n; ++it) {
      const int b = it & 1;
      if (it + 1 < n) {
        // S(it+1) once the warps hold S(it); its stage was waited for with dP
        ok = wait(s_free, it & 1, kSiteMmaSFree);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_score(0, COL_S, (it + 1) % ST, s_full);
      }
      ok = wait(&ds_ready[b], (it >> 1) & 1, kSiteMmaP);
      if (!ok) break;
      ptx::tc_fence_after();
      issue_dq(b, it % ST, it == 0);
      if (it + 2 < n) {
        const int s2 = (it + 2) % ST;
        ok = wait(&stage_full[s2], ((it + 2) / ST) & 1, kSiteMmaStage);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_score(1, COL_DP + b * 128, s2, &dp_full[b]);
      }
    }
    // every MMA issued must be complete before TMEM is freed
    if (ptx::elect_one_sync()) {
      if (ok) ptx::mma_commit(acc_full);
      ptx::mma_commit(mma_done);
    }
    __syncwarp();
    mbar_drain(mma_done, 0);
  } else {
    // ---------------------------------------------------------------- elementwise
    const int quarter = warp & 3;                    // TMEM lanes 32*quarter..
    const int half = warp >> 2;                      // keys 64*half.. of each tile
    const int row = quarter * 32 + lane;             // query row within the tile
    const int q = r0 + row;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const size_t ro = static_cast<size_t>(bh) * Tq_pad + q;  // q < Tq_pad
    const float l2 = ws_l2[ro];
    const float dd = ws_dd[ro];
    const float2 sl2 = make_float2(scale_log2, scale_log2);
    const float2 nl = make_float2(-l2, -l2);
    const float2 nd = make_float2(-dd, -dd);
    const int kmax = causal ? min(T_kv - 1, q + off) : T_kv - 1;  // last key this row sees
    bool ok = ptx::mbar_wait(res_full, 0, status, status_word(kKern, kSiteEltRes));
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      // row `row` of Q (warps 0-3) or dO (warps 4-7), from the 128-byte
      // swizzled tile (16-byte chunk c of row r sits at chunk c ^ (r % 8)),
      // into 32 TMEM columns as 16-bit pairs in K order: the A operand of the
      // score products
      const uint8_t* src = smem + (half ? OFF_DO : OFF_Q) + row * 128;
      uint32_t words[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ (row & 7)) << 4));
        words[4 * c] = v.x;
        words[4 * c + 1] = v.y;
        words[4 * c + 2] = v.z;
        words[4 * c + 3] = v.w;
      }
      ptx::tmem_st_32x32b_x32(t_lane + (half ? COL_DO : COL_Q), words);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(res_tmem);
    }
    for (int it = 0; ok && it < n; ++it) {
      const int b = it & 1;
      ok = ptx::mbar_wait(s_full, it & 1, status, status_word(kKern, kSiteEltS));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const int k0 = it * kRows + half * 64;
      const int cmax = kmax - k0;  // keys k0 + c with c <= cmax are visible
      const bool all_visible = __all_sync(0xffffffffu, cmax >= 63);
      uint32_t sr[64];
      ptx::tmem_ld_32x32b_x32(t_lane + COL_S + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      ptx::tmem_ld_32x32b_x32(t_lane + COL_S + half * 64 + 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_ld_64(sr);
      ptx::tc_fence_before();
      ptx::mbar_arrive(s_free);
      const float* s = reinterpret_cast<const float*>(sr);
      float2 pp[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float2 x = __ffma2_rn(make_float2(s[2 * j], s[2 * j + 1]), sl2, nl);
        pp[j] = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
      }
      if (!all_visible) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          pp[j].x = 2 * j <= cmax ? pp[j].x : 0.f;
          pp[j].y = 2 * j + 1 <= cmax ? pp[j].y : 0.f;
        }
      }
      ok = ptx::mbar_wait(&dp_full[b], (it >> 1) & 1, status, status_word(kKern, kSiteEltS));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_dp = t_lane + COL_DP + b * 128 + half * 64;
      uint32_t dr[64];
      ptx::tmem_ld_32x32b_x32(t_dp, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      ptx::tmem_ld_32x32b_x32(t_dp + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tmem_wait_ld_64(dr);
      const float* dp = reinterpret_cast<const float*>(dr);
      uint32_t gk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float2 g = __fmul2_rn(pp[j], __fadd2_rn(make_float2(dp[2 * j], dp[2 * j + 1]), nd));
        gk[j] = pack2<BF16>(g.x, g.y);
      }
      ptx::tmem_st_32x32b_x32(t_dp, gk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ds_ready[b]);
    }
    if (ok) {
      // -------------------------------------------------------------- epilogue
      ok = ptx::mbar_wait(acc_full, 0, status, status_word(kKern, kSiteEltAcc));
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        ptx::tc_fence_after();
        const bool write = q < T_q;
        uint8_t* dst = reinterpret_cast<uint8_t*>(dq_out) +
                       (static_cast<size_t>(bh) * T_q + (write ? q : 0)) * 64 * 2 + half * 32 * 2;
        uint32_t raw[32];
        ptx::tmem_ld_32x32b_x32(t_lane + COL_DQ + half * 32, raw);
        tmem_wait_ld_32(raw);
        if (write) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const float* f = reinterpret_cast<const float*>(&raw[g8 * 8]);
            uint4 v;
            v.x = pack2<BF16>(f[0] * scale, f[1] * scale);
            v.y = pack2<BF16>(f[2] * scale, f[3] * scale);
            v.z = pack2<BF16>(f[4] * scale, f[5] * scale);
            v.w = pack2<BF16>(f[6] * scale, f[7] * scale);
            *reinterpret_cast<uint4*>(dst + g8 * 16) = v;
          }
        }
      }
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <typename K>
cudaError_t configure_once(K kern, int smem_bytes, uint64_t* configured, int dev) {
  if (dev >= 64 || (*configured & (1ull << dev))) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess) *configured |= 1ull << dev;
  return e;
}

// The two gradient kernels of one head dimension: at d = 64 the 128-row
// streamed tiles (bwd_kv128_kernel, bwd_q128_kernel), at d = 128 bwd_kernel
// in its two modes with 64-row streamed tiles.
template <int D, bool BF16>
cudaError_t launch_bwd_t(const BwdProblem& p, cudaStream_t stream) {
  static std::mutex mu;
  static uint64_t conf_kv = 0, conf_q = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  constexpr bool k128 = D == 64;
  constexpr int kv_str = k128 ? kv128::kRows : kStr;
  constexpr int q_str = k128 ? q128::kRows : kStr;
  constexpr int kv_smem = [] {
    if constexpr (k128) return kv128::SMEM_BYTES;
    else return BwdCfg<D, true>::SMEM_BYTES;
  }();
  constexpr int q_smem = [] {
    if constexpr (k128) return q128::SMEM_BYTES;
    else return BwdCfg<D, false>::SMEM_BYTES;
  }();
  auto kern_kv = [] {
    if constexpr (k128) return bwd_kv128_kernel<BF16>;
    else return bwd_kernel<D, BF16, true>;
  }();
  auto kern_q = [] {
    if constexpr (k128) return bwd_q128_kernel<BF16>;
    else return bwd_kernel<D, BF16, false>;
  }();
  {
    std::lock_guard<std::mutex> g(mu);
    e = configure_once(kern_kv, kv_smem, &conf_kv, dev);
    if (e == cudaSuccess) e = configure_once(kern_q, q_smem, &conf_q, dev);
    if (e != cudaSuccess) return e;
  }
  const int BH = p.B * p.h;
  const int BH_kv = p.B * p.h_kv;
  const int Tq_pad = static_cast<int>(bwd_rows_padded(p.T_q));
  float* l2 = p.ws;
  float* dd = p.ws + static_cast<size_t>(BH) * Tq_pad;
  const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);

  // 1. row terms
  const long long n_rows = static_cast<long long>(BH) * Tq_pad;
  const long long rpb = 256 / (D / 8);
  bwd_prep_kernel<D, BF16><<<static_cast<unsigned>((n_rows + rpb - 1) / rpb), 256, 0, stream>>>(
      static_cast<const uint8_t*>(p.o), static_cast<const uint8_t*>(p.dout), p.lse, l2, dd, p.T_q,
      Tq_pad, n_rows);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // 2. dK, dV: resident 128-key K/V tiles, streamed Q/dO tiles
  CUtensorMap mX, mY, mU, mW;
  if (!make_map(&mX, p.k, p.T_kv, BH_kv, D, BF16, kRes) ||
      !make_map(&mY, p.v, p.T_kv, BH_kv, D, BF16, kRes) ||
      !make_map(&mU, p.q, p.T_q, BH, D, BF16, kv_str) ||
      !make_map(&mW, p.dout, p.T_q, BH, D, BF16, kv_str))
    return cudaErrorInvalidValue;
  const int n_kt = (p.T_kv + kRes - 1) / kRes;
  if constexpr (k128)
    kern_kv<<<static_cast<unsigned>(BH_kv) * n_kt, kBwdThreads, kv_smem, stream>>>(
        mX, mY, mU, mW, l2, dd, Tq_pad, p.dv, p.dk, p.T_q, p.T_kv, BH_kv, p.h, p.h_kv, p.scale,
        scale_log2, p.causal, p.status);
  else
    kern_kv<<<static_cast<unsigned>(BH_kv) * n_kt, kBwdThreads, kv_smem, stream>>>(
        mX, mY, mU, mW, l2, dd, Tq_pad, p.dv, p.dk, p.T_q, p.T_kv, BH_kv, n_kt, p.h, p.h_kv,
        p.scale, scale_log2, p.causal, p.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // 3. dQ: resident 128-row Q/dO tiles, streamed K/V tiles
  if (!make_map(&mX, p.q, p.T_q, BH, D, BF16, kRes) ||
      !make_map(&mY, p.dout, p.T_q, BH, D, BF16, kRes) ||
      !make_map(&mU, p.k, p.T_kv, BH_kv, D, BF16, q_str) ||
      !make_map(&mW, p.v, p.T_kv, BH_kv, D, BF16, q_str))
    return cudaErrorInvalidValue;
  const int n_qt = (p.T_q + kRes - 1) / kRes;
  if constexpr (k128)
    kern_q<<<static_cast<unsigned>(BH) * n_qt, kBwdThreads, q_smem, stream>>>(
        mX, mY, mU, mW, l2, dd, Tq_pad, p.dq, p.T_q, p.T_kv, BH, n_qt, p.h, p.h_kv, p.scale,
        scale_log2, p.causal, p.status);
  else
    kern_q<<<static_cast<unsigned>(BH) * n_qt, kBwdThreads, q_smem, stream>>>(
        mX, mY, mU, mW, l2, dd, Tq_pad, nullptr, p.dq, p.T_q, p.T_kv, BH, n_qt, p.h, p.h_kv,
        p.scale, scale_log2, p.causal, p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdProblem& p, cudaStream_t stream, const char** name) {
  cudaError_t e;
  if (p.d == 64) {
    e = p.bf16 ? launch_bwd_t<64, true>(p, stream) : launch_bwd_t<64, false>(p, stream);
    *name = p.bf16 ? "bwd_prep+bwd_dkdv+bwd_dq_tcgen05_d64_bf16"
                   : "bwd_prep+bwd_dkdv+bwd_dq_tcgen05_d64_f16";
  } else {
    e = p.bf16 ? launch_bwd_t<128, true>(p, stream) : launch_bwd_t<128, false>(p, stream);
    *name = p.bf16 ? "bwd_prep+bwd_dkdv+bwd_dq_tcgen05_d128_bf16"
                   : "bwd_prep+bwd_dkdv+bwd_dq_tcgen05_d128_f16";
  }
  return e;
}

}  // namespace attn
