// prefill_sm103.cu -- exact attention forward for T_q > 1 on GB300 tensor cores.
//
// One CTA owns one tile of 128 query rows of one (batch, head) and walks the
// key/value tiles of 128 keys that the tile can see:
//
//   warp 0        TMA producer: Q tile once, then K_j and V_j tiles into a
//                 multi-stage shared-memory ring (128-byte swizzle).
//   warp 1        TMEM owner and MMA issuer (one thread): S_j = Q K_j^T into a
//                 double-buffered TMEM score tile; O += P_j V_j into the TMEM
//                 output accumulator (fp32).
//   warps 2..5    softmax: thread t owns query row t (TMEM lane t). It reads
//                 its score row from TMEM, applies the causal/tail mask,
//                 updates the running max m and running sum l, writes
//                 P_j = exp(scale*S_j - m) as 16-bit into shared memory for
//                 the PV product, rescales its O row in TMEM when m has to
//                 move, and finally writes O = o/l and lse = m + ln l.
//
// The score and probability tiles live only in TMEM, registers and shared
// memory; O is written to HBM once. This is the tiled forward of
// "FlashAttention IO-aware tiling lab" ("Read each kernel phase": load Q,
// score a K tile, update the online softmax, accumulate V, write O once) and
// the recurrence of "IO-Aware Attention: Tiling the Score Matrix Without
// Materializing It", section "Softmax over blocks, exactly". Causal tiles
// beyond the diagonal are never loaded or computed and only tiles that
// straddle it are masked (same page, section "Parallelism and the cost of
// the split", last paragraph). Accumulation and rescaling are fp32 (same
// page, section "Where the approach stops helping", last paragraph).
//
// Differences from the pages' sketch, for sm_103a: accumulators live in
// TMEM instead of registers/shared memory, so the 128 x d accumulator no
// longer bounds the tile; the running max is moved lazily -- a row keeps its
// old reference max until the new one exceeds it by 2^8 (in exp2 units), so
// P stays <= 256 and the O rescale is rare. Because o and l share one
// reference, o/l is unchanged: the result is still exact up to rounding.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace attn {

namespace {

constexpr int kBM = 128;       // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;       // keys per K/V tile
constexpr int kSub = 128 * 128;  // bytes of one [128 rows][64 x 16-bit] swizzled sub-tile
constexpr int kThreads = 192;  // 6 warps
constexpr float kRebaseLog2 = 8.0f;  // lazy rescale threshold (P <= 2^8)

template <int D>
struct Cfg {
  static constexpr int STAGES = (D == 64) ? 3 : 2;
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int KV_BYTES = kBN * D * 2;
  static constexpr int P_BYTES = kBM * kBN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S],
  // s_full[2], s_empty[2], p_full[2], p_empty[2], o_done, mma_done
  static constexpr int N_BARS = 1 + 4 * STAGES + 8 + 2;
  static constexpr int OFF_TMEMPTR = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
};

// Wait sites recorded in the status word on a timeout.
enum : uint32_t {
  kSiteProdKEmpty = 1, kSiteProdVEmpty, kSiteMmaQ, kSiteMmaK, kSiteMmaSEmpty, kSiteMmaV,
  kSiteMmaP, kSiteSoftS, kSiteSoftPEmpty, kSiteSoftO, kSiteEpiO, kSiteMmaDone
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

// tcgen05.wait::ld that also ties the loaded registers to the wait, so no
// use of them can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// Bounded wait used only while draining after an error: ignores the
// status word, gives up after the same time limit.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = ptx::smem_u32(bar);
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(a, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, void* __restrict__ out,
                   float* __restrict__ lse, int T_q, int T_kv, int BH, int n_qtiles,
                   float scale_log2, int causal, unsigned int* __restrict__ status) {
  using C = Cfg<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + ST;
  uint64_t* v_full = k_empty + ST;
  uint64_t* v_empty = v_full + ST;
  uint64_t* s_full = v_empty + ST;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 2;
  uint64_t* o_done = p_empty + 2;
  uint64_t* mma_done = o_done + 1;
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMPTR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heaviest query tiles first (largest index under a causal mask), all
  // heads of one tile index before the next: the block scheduler then hands
  // out the long tiles early and the short ones fill the tail.
  const int qt = n_qtiles - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int q0 = qt * kBM;
  const int off = T_kv - T_q;
  int kv_end = T_kv;
  if (causal) {
    const int last_row = min(q0 + kBM - 1, T_q - 1);
    kv_end = min(T_kv, last_row + off + 1);
  }
  const int n_kv = (kv_end + kBN - 1) / kBN;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int i = 0; i < ST; ++i) {
      ptx::mbar_init(&k_full[i], 1);
      ptx::mbar_init(&k_empty[i], 1);
      ptx::mbar_init(&v_full[i], 1);
      ptx::mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s_full[i], 1);
      ptx::mbar_init(&s_empty[i], 128);
      ptx::mbar_init(&p_full[i], 128);
      ptx::mbar_init(&p_empty[i], 1);
    }
    ptx::mbar_init(o_done, 1);
    ptx::mbar_init(mma_done, 1);
    ptx::fence_mbarrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_ptr, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  const uint32_t sQ = ptx::smem_u32(smem + C::OFF_Q);
  const uint32_t sK = ptx::smem_u32(smem + C::OFF_K);
  const uint32_t sV = ptx::smem_u32(smem + C::OFF_V);
  const uint32_t sP = ptx::smem_u32(smem + C::OFF_P);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmQ);
      ptx::prefetch_tensormap(&tmK);
      ptx::prefetch_tensormap(&tmV);
      const uint64_t pol_kv = ptx::policy_evict_last();
      const uint64_t pol_q = ptx::policy_evict_first();
      ptx::mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        ptx::tma_load_3d(smem + C::OFF_Q + c * kSub, &tmQ, q_full, c * 64, q0, bh, pol_q);
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j % ST;
        const uint32_t ph = (j / ST) & 1;
        ok = ptx::mbar_wait(&k_empty[st], ph ^ 1, status, status_word(kKernPrefill, kSiteProdKEmpty));
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          ptx::tma_load_3d(smem + C::OFF_K + st * C::KV_BYTES + c * kSub, &tmK, &k_full[st],
                           c * 64, j * kBN, bh, pol_kv);
        k_issued = j + 1;
        ok = ptx::mbar_wait(&v_empty[st], ph ^ 1, status, status_word(kKernPrefill, kSiteProdVEmpty));
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          ptx::tma_load_3d(smem + C::OFF_V + st * C::KV_BYTES + c * kSub, &tmV, &v_full[st],
                           c * 64, j * kBN, bh, pol_kv);
        v_issued = j + 1;
      }
      if (!ok) {
        // Error path: let the copies already in flight land before the CTA
        // (and its shared memory) goes away. Only the last STAGES loads of
        // each ring can still be outstanding.
        mbar_drain(q_full, 0);
        for (int j = max(0, k_issued - ST); j < k_issued; ++j) mbar_drain(&k_full[j % ST], (j / ST) & 1);
        for (int j = max(0, v_issued - ST); j < v_issued; ++j) mbar_drain(&v_full[j % ST], (j / ST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = ptx::make_idesc_f16(BF16, kBM, kBN, false, false);
      constexpr uint32_t idO = ptx::make_idesc_f16(BF16, kBM, D, false, true);
      bool ok = ptx::mbar_wait(q_full, 0, status, status_word(kKernPrefill, kSiteMmaQ));
      for (int j = 0; j <= n_kv && ok; ++j) {
        if (j < n_kv) {
          const int st = j % ST;
          const int sb = j & 1;
          ok = ptx::mbar_wait(&k_full[st], (j / ST) & 1, status, status_word(kKernPrefill, kSiteMmaK));
          if (!ok) break;
          ok = ptx::mbar_wait(&s_empty[sb], ((j >> 1) & 1) ^ 1, status,
                              status_word(kKernPrefill, kSiteMmaSEmpty));
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t kbase = sK + st * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kSub + (kk & 3) * 32;
            const uint64_t a = ptx::make_sdesc_sw128(sQ + koff, 16, 1024);
            const uint64_t b = ptx::make_sdesc_sw128(kbase + koff, 16, 1024);
            ptx::mma_f16_ss(tmem + (sb ? C::COL_S1 : C::COL_S0), a, b, idS, kk > 0);
          }
          ptx::mma_commit(&s_full[sb]);
          ptx::mma_commit(&k_empty[st]);
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int st = jj % ST;
          const int pb = jj & 1;
          ok = ptx::mbar_wait(&v_full[st], (jj / ST) & 1, status, status_word(kKernPrefill, kSiteMmaV));
          if (!ok) break;
          ok = ptx::mbar_wait(&p_full[pb], (jj >> 1) & 1, status, status_word(kKernPrefill, kSiteMmaP));
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t vbase = sV + st * C::KV_BYTES;
          const uint32_t pbase = sP + pb * C::P_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t a =
                ptx::make_sdesc_sw128(pbase + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
            const uint64_t b = ptx::make_sdesc_sw128(vbase + kk * 16 * 128, kSub, 1024);
            ptx::mma_f16_ss(tmem + C::COL_O, a, b, idO, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(o_done);
          ptx::mma_commit(&v_empty[st]);
          ptx::mma_commit(&p_empty[pb]);
        }
      }
      // All MMAs this thread issued must be complete before TMEM is freed.
      ptx::mma_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;               // TMEM lanes [32*quarter, 32*quarter+32)
    const int r = quarter * 32 + lane;          // row within the tile
    const int row = q0 + r;                     // absolute query row
    const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int last_key = causal ? min(T_kv - 1, row + off) : T_kv - 1;
    float m_used = -INFINITY;  // reference max, log2 units of the scaled score
    float l = 0.f;
    bool ok = true;
    uint8_t* prow_base = smem + C::OFF_P + r * 128;
    const int rsw = r & 7;

    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      const int pb = j & 1;
      ok = ptx::mbar_wait(&s_full[sb], (j >> 1) & 1, status, status_word(kKernPrefill, kSiteSoftS));
      // tcgen05.ld/st/wait are warp-collective (.sync.aligned): every branch
      // around them must be taken by the whole warp.
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t raw[32];
        ptx::tmem_ld_32x32b_x32(t_row + (sb ? C::COL_S1 : C::COL_S0) + c * 32, raw);
        tmem_wait_ld_regs(raw);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw[i]);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s_empty[sb]);

      const int key0 = j * kBN;
      if (key0 + kBN - 1 > last_key) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (key0 + c > last_key) s[c] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; ++c) mx = fmaxf(mx, s[c]);
      const float m_tile = mx * scale_log2;
      float alpha = 1.f;
      bool rescale = false;
      if (m_tile > m_used + kRebaseLog2) {
        alpha = ptx::ex2_approx(m_used - m_tile);   // 0 when m_used = -inf
        rescale = (m_used != -INFINITY);
        l *= alpha;
        m_used = m_tile;
      }
      const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;

      ok = ptx::mbar_wait(&p_empty[pb], ((j >> 1) & 1) ^ 1, status,
                          status_word(kKernPrefill, kSiteSoftPEmpty));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      float rs = 0.f;
      uint8_t* prow = prow_base + pb * C::P_BYTES;
#pragma unroll
      for (int c = 0; c < kBN / 8; ++c) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          p[i] = ptx::ex2_approx(fmaf(s[c * 8 + i], scale_log2, -m_ref));
          rs += p[i];
        }
        uint4 w;
        w.x = pack2<BF16>(p[0], p[1]);
        w.y = pack2<BF16>(p[2], p[3]);
        w.z = pack2<BF16>(p[4], p[5]);
        w.w = pack2<BF16>(p[6], p[7]);
        const int sub = c >> 3;   // keys 0-63 / 64-127
        const int chunk = (c & 7) ^ rsw;
        *reinterpret_cast<uint4*>(prow + sub * kSub + (chunk << 4)) = w;
      }
      l += rs;
      ptx::fence_proxy_async_smem();

      if (__any_sync(0xffffffffu, rescale)) {
        // O holds the sum through tile j-1; wait for that product, then
        // multiply this warp's rows of O by their alpha in place (rows that
        // keep their reference max have alpha = 1).
        ok = ptx::mbar_wait(o_done, (j - 1) & 1, status, status_word(kKernPrefill, kSiteSoftO));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        const float mul = rescale ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t raw[32];
          ptx::tmem_ld_32x32b_x32(t_row + C::COL_O + c * 32, raw);
          tmem_wait_ld_regs(raw);
#pragma unroll
          for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * mul);
          ptx::tmem_st_32x32b_x32(t_row + C::COL_O + c * 32, raw);
        }
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&p_full[pb]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok) ok = ptx::mbar_wait(o_done, (n_kv - 1) & 1, status, status_word(kKernPrefill, kSiteEpiO));
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      ptx::tc_fence_after();
      const float inv_l = 1.f / l;
      const bool write = row < T_q;
      uint8_t* orow = reinterpret_cast<uint8_t*>(out) +
                      (static_cast<size_t>(bh) * T_q + (write ? row : 0)) * D * 2;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t raw[32];
        ptx::tmem_ld_32x32b_x32(t_row + C::COL_O + c * 32, raw);
        tmem_wait_ld_regs(raw);
        if (write) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 w;
            w.x = pack2<BF16>(__uint_as_float(raw[g * 8 + 0]) * inv_l, __uint_as_float(raw[g * 8 + 1]) * inv_l);
            w.y = pack2<BF16>(__uint_as_float(raw[g * 8 + 2]) * inv_l, __uint_as_float(raw[g * 8 + 3]) * inv_l);
            w.z = pack2<BF16>(__uint_as_float(raw[g * 8 + 4]) * inv_l, __uint_as_float(raw[g * 8 + 5]) * inv_l);
            w.w = pack2<BF16>(__uint_as_float(raw[g * 8 + 6]) * inv_l, __uint_as_float(raw[g * 8 + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + (c * 32 + g * 8) * 2) = w;
          }
        }
      }
      if (write)
        lse[static_cast<size_t>(bh) * T_q + row] = (m_used + __log2f(l)) * 0.69314718055994531f;
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// [BH][T][D] 16-bit tensor viewed as 3-D (D innermost), box 64 x 128 x 1,
// 128-byte swizzle; rows past T read as zero.
bool make_map(CUtensorMap* map, const void* base, int T, int BH, int D, bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool BF16>
cudaError_t launch_t(const FwdProblem& p, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = prefill_kernel<D, BF16>;
  static std::mutex mu;
  static uint64_t configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64 && !(configured & (1ull << dev))) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      configured |= 1ull << dev;
    }
  }
  const int BH = p.B * p.h;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.T_q, BH, D, BF16) || !make_map(&mk, p.k, p.T_kv, BH, D, BF16) ||
      !make_map(&mv, p.v, p.T_kv, BH, D, BF16))
    return cudaErrorInvalidValue;
  const int n_qtiles = (p.T_q + kBM - 1) / kBM;
  const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
  dim3 grid(static_cast<unsigned>(n_qtiles) * static_cast<unsigned>(BH));
  kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(mq, mk, mv, p.o, p.lse, p.T_q, p.T_kv, BH,
                                                  n_qtiles, scale_log2, p.causal, p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const FwdProblem& p, cudaStream_t stream, const char** name) {
  cudaError_t e;
  if (p.d == 64) {
    e = p.bf16 ? launch_t<64, true>(p, stream) : launch_t<64, false>(p, stream);
    *name = p.bf16 ? "prefill_tcgen05_d64_bf16" : "prefill_tcgen05_d64_f16";
  } else {
    e = p.bf16 ? launch_t<128, true>(p, stream) : launch_t<128, false>(p, stream);
    *name = p.bf16 ? "prefill_tcgen05_d128_bf16" : "prefill_tcgen05_d128_f16";
  }
  return e;
}

}  // namespace attn
