// prefill_sm103.cu -- exact attention forward for T_q > 1 on GB300 tensor cores
// (also the grouped-query and paged decode of groups >= 4, as prefills of G
// query rows per key/value head).
//
// A persistent CTA owns a sequence of work units. A unit is two 128-row
// query tiles, A and B: rows [q0, q0+128) and [q0+128, q0+256) of one head
// sharing one stream of 128-key K/V tiles (row pairs), or, for at most 128
// query rows at d = 64, the rows of two heads with a K/V stream each (head
// pairs). With S > 1 a unit covers one key partition and writes fp32
// partials (o, m, l) for the merge kernel instead of O and lse. Roles (384
// threads, three warpgroups):
//
//   warps 0-3     softmax of tile A; thread t owns query row t (TMEM lane t)
//   warps 4-7     softmax of tile B
//   warp 8        TMA producer: Q_A, Q_B once per unit, then K and V tiles into
//                 a ring of shared-memory slots (128-byte swizzle); one lane,
//                 or the whole warp with a paged cache (lane i gathers box i)
//   warp 9        TMEM owner and MMA issuer (elected lane, warp-uniform loop);
//                 at d = 64 it issues tile A's products and warp 10 tile B's
//   warps 10-11   otherwise no role; their warpgroup hands its registers to
//                 the softmax warpgroups
//
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A and O_B after
// them (d columns each); at d = 64 P_A and P_B have columns of their own
// after O, at d = 128 P_X overwrites the first 64 columns of S_X. S_X = Q_X
// K_j^T is a tcgen05.mma chain (M=128, N=128) from shared memory; the softmax
// warps turn it into P_X = 2^(scale*log2e*S_X - m) as 16-bit values; O_X +=
// P_X V_j reads P from tensor memory and V from shared memory. The tensor
// core works on one tile while the other tile's softmax runs. At d = 128 one
// thread issues both tiles in the order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1),
// so S_X(j+1) overwrites P_X(j) only after PV_X(j) read it; at d = 64 each
// tile's issuer starts S_X(j+1) as soon as its softmax has loaded S_X(j).
//
// Scores and probabilities never leave the chip; O is written to HBM once.
// This is the tiled forward of "FlashAttention IO-aware tiling lab" ("Read
// each kernel phase": load Q, score a K tile, update the online softmax,
// accumulate V, write O once) with the recurrence of "IO-Aware Attention:
// Tiling the Score Matrix Without Materializing It", section "Softmax over
// blocks, exactly". Causal units stop their key loop at the diagonal and
// only tiles crossing it are masked (same page, section "Parallelism and the
// cost of the split", last paragraph). Accumulation and rescaling are fp32
// (same page, section "Where the approach stops helping").
//
// sm_103a-specific choices: accumulators in TMEM (the 128 x d accumulator
// does not bound the tile); a lazy running max -- a row keeps its reference
// max until a new score exceeds it by 2^8, so P <= 256 and O is rarely
// rescaled (o and l share the reference, so o/l is unchanged); packed fp32x2
// arithmetic in the softmax; and an MMA issuer that builds its shared-memory
// descriptors once and issues fully unrolled chains (a rolled loop with
// per-MMA descriptor arithmetic made the single issuing thread, not the
// tensor core, the bottleneck: ~83 vs ~45-64 cycles per MMA).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "attn_status.h"
#include "ptx_sm103.cuh"
#include "tma_host.h"

namespace attn {

namespace {

constexpr int kBM = 128;          // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kSub = 128 * 128;   // bytes of one [128 rows][64 x 16-bit] swizzled sub-tile
constexpr int kThreads = 384;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
// Register split (setmaxnreg): the launch gives 384 x 168 = 64512 registers;
// the two softmax warpgroups take 200 each per thread and the control
// warpgroup keeps 104: 2 x 128 x 200 + 128 x 104 = 64512 <= 64512.
constexpr int kRegsSoftmax = 200;
constexpr int kRegsControl = 104;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl <= kThreads * 168, "register split");
constexpr float kRebaseLog2 = 8.0f;  // lazy rescale threshold (P <= 2^8)

template <int D>
struct Cfg {
  static constexpr int TILE_BYTES = kBM * D * 2;   // one Q, K or V tile
  static constexpr int SLOTS = (D == 64) ? 10 : 5;
  static constexpr int OFF_Q = 0;                  // Q_A, Q_B
  static constexpr int OFF_RING = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_RING + SLOTS * TILE_BYTES;
  // q_full, q_empty, slot_full[S], slot_empty[S], s_full[2], p_full[2],
  // o_full[2], o_empty[2], mma_done, s_free[2], pv_done[2]
  static constexpr int N_BARS = 2 + 2 * SLOTS + 8 + 1 + 4;
  static constexpr int OFF_TMEMPTR = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  // d = 64 leaves TMEM room (S 2x128 + O 2x64 = 384 columns) for P in
  // columns of its own (2x64): S_X(j+1) can then be computed as soon as the
  // softmax has read S_X(j), while P_X(j) and PV_X(j) are still in flight,
  // which takes the MMA issue of PV_X(j) and S_X(j+1) off the softmax's
  // critical path. d = 128 fills TMEM with S and O, and P overwrites S.
  static constexpr bool SEP_P = (D == 64);
};

// Head pairs with a paged cache: at the start of each unit the producer
// copies the unit's block-table entries (per tile, the pages its key range
// touches) into shared memory, so the page of every box is a shared-memory
// read, not a dependent global load per box in the producer's path. Both
// tiles' entries are loaded in one pass, four per lane in flight (one table
// round trip per unit instead of one per 32 entries and tile: 64-row pages
// 194 -> 189 us for 32 sequences x 16K keys). (Copying the next unit's
// entries ahead of time was measured slower.) Key ranges that need more
// entries than the buffer holds read the table per box instead.
constexpr int kTblEntries = 2048;
constexpr int kTblBytes = 2 * kTblEntries * 4;  // [tile][entry]

__host__ __device__ constexpr uint32_t col_s(int x) { return static_cast<uint32_t>(x) * 128u; }
template <int D>
__host__ __device__ constexpr uint32_t col_o(int x) {
  return 256u + static_cast<uint32_t>(x) * static_cast<uint32_t>(D);
}
// P_X when it has columns of its own (SEP_P): after O_A and O_B
__host__ __device__ constexpr uint32_t col_p(int x) { return 384u + static_cast<uint32_t>(x) * 64u; }

// Wait sites recorded in the status word on a timeout.
enum : uint32_t {
  kSiteProdQ = 1, kSiteProdSlot, kSiteMmaQ, kSiteMmaSlot, kSiteMmaP, kSiteMmaOEmpty,
  kSiteSoftS, kSiteSoftO, kSiteMmaSFree, kSiteSoftPv, kSiteBadPage
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

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Four tcgen05.ld of 32 columns each, then one wait that is tied to all 128
// registers so no use of them can be scheduled before the data arrives.
__device__ __forceinline__ void tmem_ld_row128(uint32_t taddr, uint32_t (&r)[128]) {
  ptx::tmem_ld_32x32b_x32(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  ptx::tmem_ld_32x32b_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  ptx::tmem_ld_32x32b_x32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
  ptx::tmem_ld_32x32b_x32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
#define R8(b) "+r"(r[b]), "+r"(r[b + 1]), "+r"(r[b + 2]), "+r"(r[b + 3]), "+r"(r[b + 4]), \
              "+r"(r[b + 5]), "+r"(r[b + 6]), "+r"(r[b + 7])
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : R8(0), R8(8), R8(16), R8(24), R8(32), R8(40), R8(48), R8(56), R8(64), R8(72),
                 R8(80), R8(88), R8(96), R8(104), R8(112), R8(120)
               :
               : "memory");
#undef R8
}

// tcgen05.wait::ld tied to 32 registers.
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

// An empty statement tied to registers. The softmax arithmetic is register
// work, which the compiler may otherwise move across the barrier waits
// (volatile asm orders only against other volatile asm and memory): the
// fence keeps the computation of these values before the waits after it.
__device__ __forceinline__ void reg_fence64f(uint32_t (&r)[64], float& f) {
#define R8(b) "+r"(r[b]), "+r"(r[b + 1]), "+r"(r[b + 2]), "+r"(r[b + 3]), "+r"(r[b + 4]), \
              "+r"(r[b + 5]), "+r"(r[b + 6]), "+r"(r[b + 7])
  asm volatile("" : R8(0), R8(8), R8(16), R8(24), R8(32), R8(40), R8(48), R8(56), "+f"(f));
#undef R8
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

// One work unit: query tiles A and B and key partition s of S: key tiles
// [j0, j0 + n_all), of which tile A sees the first n_a and tile B the first
// n_b (causal: up to the diagonal). Row-pair mode: A = rows [q0, q0+128) and
// B = [q0+128, q0+256) of one head, reading one K/V stream. Head-pair mode
// (at most 128 query rows, d = 64): A = the rows of head bh and B = those of
// head bh + 1, each reading its own K/V stream, so that the two tiles that
// keep the tensor core and the softmax warps busy in turn both exist for
// short queries (grouped-query decode, short prefill); rows_b = 0 when bh is
// the last head. With S = 1 the partition is every key tile the tiles see.
struct Unit {
  int bh, kvbh, q0, tkv;          // tile A: head, key/value head, first row, keys
  int bh_b, kvbh_b, q0_b, tkv_b;  // tile B
  int rows_b, n_a, n_b, n_all, j0, s;
};

// Keys from a paged pool ([num_pages][h_kv][page_size][d]) through a block
// table (int32 [B][max_pages]) with per-sequence lengths: the mode that runs
// grouped-query decode against a paged cache (virtual head bh = b*h_kv + kv
// head, its G query heads as query rows). table == nullptr: contiguous K/V.
struct PagedKV {
  const int* table;
  const int* lens;
  int page_shift, max_pages, num_pages;
};

template <bool HP>
__device__ __forceinline__ Unit unit_info(int u, int BH, int n_pairs, int T_q, int T_kv,
                                          int causal, int h_q, int h_kv, int S, const int* lens) {
  Unit w;
  w.s = u % S;
  u /= S;
  // paged mode: a sequence's length (b = bh / h_q), clamped to what its table
  // can name (T_kv); otherwise every head has T_kv keys
  auto keys_of = [&](int bh) { return lens ? max(0, min(__ldg(lens + bh / h_q), T_kv)) : T_kv; };
  // grouped-query attention: query head i reads key/value head i / (h_q / h_kv)
  auto kv_of = [&](int bh) { return (bh / h_q) * h_kv + (bh % h_q) / (h_q / h_kv); };
  int rows_a;
  if constexpr (HP) {
    w.bh = 2 * u;
    w.bh_b = w.bh + 1;
    w.q0 = 0;
    w.q0_b = 0;
    rows_a = T_q;
    w.rows_b = w.bh_b < BH ? T_q : 0;
  } else {
    const int pair = n_pairs - 1 - u / BH;  // heaviest pairs first under a causal mask
    w.bh = u % BH;
    w.bh_b = w.bh;
    w.q0 = pair * 2 * kBM;
    w.q0_b = w.q0 + kBM;
    rows_a = min(kBM, T_q - w.q0);
    w.rows_b = max(0, min(kBM, T_q - w.q0_b));
  }
  w.tkv = keys_of(w.bh);
  w.kvbh = kv_of(w.bh);
  w.tkv_b = HP && w.rows_b > 0 ? keys_of(w.bh_b) : w.tkv;
  w.kvbh_b = HP && w.rows_b > 0 ? kv_of(w.bh_b) : w.kvbh;
  const int off = T_kv - T_q;  // causal alignment (the paged mode is never causal)
  auto n_tiles = [&](int keys, int last_row) {
    const int n_kv = (keys + kBN - 1) / kBN;
    return causal ? min(n_kv, (last_row + off + kBN) / kBN) : n_kv;
  };
  w.n_a = n_tiles(w.tkv, w.q0 + rows_a - 1);
  w.n_b = w.rows_b > 0 ? n_tiles(w.tkv_b, w.q0_b + w.rows_b - 1) : 0;
  // key partition s of S: ceil(N/S) key tiles each, N = the unit's key tiles
  const int n_full = max(w.n_a, w.n_b);
  const int chunk = (n_full + S - 1) / S;
  w.j0 = w.s * chunk;
  const int span = max(0, min(n_full, w.j0 + chunk) - w.j0);
  w.n_a = max(0, min(w.n_a - w.j0, span));
  w.n_b = max(0, min(w.n_b - w.j0, span));
  w.n_all = max(w.n_a, w.n_b);
  return w;
}

// Unit visited in round r by CTA bid of G: snake order over the heaviest-first
// list, so that a CTA that took a heavy unit in one round takes a light one in
// the next.
__device__ __forceinline__ int unit_of_round(int r, int bid, int G) {
  return (r & 1) ? r * G + (G - 1 - bid) : r * G + bid;
}

// HP: head-pair mode (two heads per unit, d = 64 only).
template <int D, bool BF16, bool PAGED, bool HP>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, void* __restrict__ out,
                   float* __restrict__ lse, int T_q, int T_kv, int BH, int n_pairs,
                   float scale_log2, int causal, unsigned int* __restrict__ status, int h_q,
                   int h_kv, int S, float* __restrict__ part, const PagedKV pkv) {
  static_assert(!HP || D == 64, "head pairs: d = 64");
  using C = Cfg<D>;
  constexpr int SL = C::SLOTS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* slot_full = bars + 2;
  uint64_t* slot_empty = slot_full + SL;
  uint64_t* s_full = slot_empty + SL;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* o_empty = o_full + 2;
  uint64_t* mma_done = o_empty + 2;
  uint64_t* s_free = mma_done + 1;   // SEP_P: softmax X has read S_X (128 arrivals)
  uint64_t* pv_done = s_free + 2;    // SEP_P: PV_X complete (P_X and O_X free)
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMPTR);
  // (paged head pairs only) the staged block-table entries of tiles A and B
  int* tbl = reinterpret_cast<int*>(smem + C::OFF_TMEMPTR + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // units: (query-tile pair, head, key partition), or (head pair, key
  // partition) in head-pair mode; S > 1 writes fp32 partials (o, m, l) to
  // `part` for the merge kernel instead of O and lse
  const int U = (HP ? (BH + 1) / 2 : n_pairs * BH) * S;
  const int G = static_cast<int>(gridDim.x);
  const int bid = static_cast<int>(blockIdx.x);
  const int off = T_kv - T_q;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    // released by each MMA-issuing warp (two at d = 64: one per tile)
    ptx::mbar_init(q_empty, C::SEP_P ? 2 : 1);
    for (int i = 0; i < SL; ++i) {
      ptx::mbar_init(&slot_full[i], 1);
      ptx::mbar_init(&slot_empty[i], C::SEP_P ? 2 : 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(&s_full[x], 1);
      ptx::mbar_init(&p_full[x], 128);
      ptx::mbar_init(&o_full[x], 1);
      ptx::mbar_init(&o_empty[x], 128);
    }
    ptx::mbar_init(mma_done, C::SEP_P ? 2 : 1);
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(&s_free[x], 128);
      ptx::mbar_init(&pv_done[x], 1);
    }
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

  // Each setmaxnreg sits in the branch of the role code it serves, so the
  // compiler applies its register limit to exactly that code.
  if (warp >= 8) {
    // one setmaxnreg instruction for the whole control warpgroup (.aligned)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == kWarpProducer) {
      // ------------------------------------------------------------ producer
      // One lane, except with a paged cache: there the whole warp runs the
      // loop (its waits made warp-uniform) and lane i looks up and loads box
      // i of each key tile, so a tile's table reads and copies run side by
      // side instead of one after another.
      if (PAGED || lane == 0) {
        const bool lead = lane == 0;
        auto uniform = [&](bool v) -> bool {
          if constexpr (PAGED) return __all_sync(0xffffffffu, v) != 0;
          return v;
        };
        if (lead) {
          ptx::prefetch_tensormap(&tmQ);
          ptx::prefetch_tensormap(&tmK);
          ptx::prefetch_tensormap(&tmV);
        }
        const uint64_t pol_kv = ptx::policy_evict_last();
        const uint64_t pol_q = ptx::policy_evict_first();
        uint32_t g = 0;   // ring fills issued
        uint32_t nq = 0;  // Q loads issued
        bool ok = true;
        for (int r = 0; ok && r * G < U; ++r) {
          const int u = unit_of_round(r, bid, G);
          if (u >= U) continue;
          const Unit w = unit_info<HP>(u, BH, n_pairs, T_q, T_kv, causal, h_q, h_kv, S, pkv.lens);
          if (w.n_all == 0) continue;  // a key partition the pair does not reach
          ok = uniform(ptx::mbar_wait(q_empty, (nq & 1) ^ 1, status,
                                      status_word(kKernPrefill, kSiteProdQ)));
          if (!ok) break;
          if (lead) {
            ptx::mbar_arrive_expect_tx(q_full, C::TILE_BYTES * (w.rows_b > 0 ? 2 : 1));
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
              ptx::tma_load_3d(smem + C::OFF_Q + c * kSub, &tmQ, q_full, c * 64, w.q0, w.bh, pol_q);
              if (w.rows_b > 0)
                ptx::tma_load_3d(smem + C::OFF_Q + C::TILE_BYTES + c * kSub, &tmQ, q_full, c * 64,
                                 w.q0_b, w.bh_b, pol_q);
            }
          }
          ++nq;
          if constexpr (!HP) {
            // one stream for both tiles: K_j, V_j
            for (int j = 0; ok && j < w.n_all; ++j) {
              int pg = 0;  // paged: this lane's box of key tile j (shared by K_j and V_j)
#pragma unroll
              for (int kind = 0; kind < 2; ++kind) {  // K_j, then V_j
                const uint32_t slot = g % SL;
                ok = uniform(ptx::mbar_wait(&slot_empty[slot], ((g / SL) & 1) ^ 1, status,
                                            status_word(kKernPrefill, kSiteProdSlot)));
                if (!ok) break;
                if (lead) ptx::mbar_arrive_expect_tx(&slot_full[slot], C::TILE_BYTES);
                uint8_t* dst = smem + C::OFF_RING + slot * C::TILE_BYTES;
                if constexpr (PAGED) {
                  // the tile's 128 keys in boxes of min(page_size, 128) rows,
                  // box i from the page the table names, by lane i (rows past
                  // the length: page 0, masked later; a bad entry is
                  // reported, never dereferenced). The copies start after the
                  // lead lane has announced the tile's bytes.
                  __syncwarp();
                  const int rows = min(1 << pkv.page_shift, kBN);
                  const int b = w.bh / h_q;  // sequence of this virtual head
                  const int kvh = w.bh - b * h_q;
                  const int i = lane * rows;
                  const int key = (w.j0 + j) * kBN + i;
                  if (i < kBN) {
                    if (kind == 0) {
                      pg = 0;
                      if (key < w.tkv) {
                        pg = __ldg(pkv.table + static_cast<size_t>(b) * pkv.max_pages +
                                   (key >> pkv.page_shift));
                        if (static_cast<unsigned>(pg) >= static_cast<unsigned>(pkv.num_pages)) {
                          atomicCAS(status, 0u,
                                    status_word_code(1u /* ATTN_ERR_INVALID_ARG */, kKernPrefill,
                                                     kSiteBadPage));
                          pg = 0;
                        }
                      }
                    }
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                      ptx::tma_load_3d(dst + c * kSub + i * 128, kind ? &tmV : &tmK,
                                       &slot_full[slot], c * 64, key & ((1 << pkv.page_shift) - 1),
                                       pg * h_q + kvh, pol_kv);
                  }
                } else {
#pragma unroll
                  for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d(dst + c * kSub, kind ? &tmV : &tmK, &slot_full[slot], c * 64,
                                     (w.j0 + j) * kBN, w.kvbh, pol_kv);
                }
                ++g;
              }
            }
          } else {
            // a stream per tile: K_j of A, K_j of B, V_j of A, V_j of B. Each
            // slot is read by one tile; this thread stands in for the release
            // of the other (slot_empty counts two), and for both when the
            // tile it belongs to has no key tile j (then the slot gets no data
            // and its full barrier just completes, keeping the phases in step).
            const int nt = w.rows_b > 0 ? 2 : 1;
            if constexpr (PAGED) {
              // Paged cache: the whole warp runs this loop (waits made
              // warp-uniform); lane i copies box i of each key tile. First
              // the unit's table entries: for tile t, the pages holding keys
              // [j0 * kBN, min(length, (j0 + n_t) * kBN)) -- only entries a
              // valid key uses are read (and checked).
              int p_lo[2] = {0, 0};
              int cnt0 = 0, cnt1 = 0;  // entries of tiles A and B
              const int* row0 = pkv.table;
              const int* row1 = pkv.table;
              bool staged = true;
              for (int t = 0; t < nt; ++t) {
                const int n_t = t ? w.n_b : w.n_a;
                const int b = (t ? w.bh_b : w.bh) / h_q;
                const int k_end = min(t ? w.tkv_b : w.tkv, (w.j0 + n_t) * kBN);
                const int lo = (w.j0 * kBN) >> pkv.page_shift;
                const int cnt = k_end > w.j0 * kBN ? ((k_end - 1) >> pkv.page_shift) + 1 - lo : 0;
                p_lo[t] = lo;
                const int* row = pkv.table + static_cast<size_t>(b) * pkv.max_pages + lo;
                if (t) {
                  cnt1 = cnt;
                  row1 = row;
                } else {
                  cnt0 = cnt;
                  row0 = row;
                }
                if (cnt > kTblEntries) staged = false;
              }
              // both tiles' entries in one pass, four loads per lane in flight
              // (entry e: tile 0's e-th, or tile 1's (e - count of tile 0)-th)
              const int total = staged ? cnt0 + cnt1 : 0;
              for (int e0 = 0; e0 < total; e0 += 128) {
                int pgs[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int e = e0 + u * 32 + lane;
                  pgs[u] = e < total ? __ldg(e < cnt0 ? row0 + e : row1 + (e - cnt0)) : 0;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int e = e0 + u * 32 + lane;
                  if (e < total) {
                    const int t = e < cnt0 ? 0 : 1;
                    int pg = pgs[u];
                    if (static_cast<unsigned>(pg) >= static_cast<unsigned>(pkv.num_pages)) {
                      atomicCAS(status, 0u,
                                status_word_code(1u /* ATTN_ERR_INVALID_ARG */, kKernPrefill,
                                                 kSiteBadPage));
                      pg = 0;
                    }
                    tbl[t * kTblEntries + (e - t * cnt0)] = pg;
                  }
                }
              }
              __syncwarp();
              const int rows = min(1 << pkv.page_shift, kBN);
              for (int j = 0; ok && j < w.n_all; ++j) {
                for (int kind = 0; ok && kind < 2; ++kind) {
                  for (int t = 0; ok && t < nt; ++t) {
                    const uint32_t slot = g % SL;
                    ok = uniform(ptx::mbar_wait(&slot_empty[slot], ((g / SL) & 1) ^ 1, status,
                                                status_word(kKernPrefill, kSiteProdSlot)));
                    if (!ok) break;
                    const bool skip = j >= (t ? w.n_b : w.n_a);
                    if (skip) {
                      // no data: the full barrier just completes, and this
                      // thread releases the slot for both tiles
                      if (lead) {
                        ptx::mbar_arrive(&slot_full[slot]);
                        ptx::mbar_arrive(&slot_empty[slot]);
                        ptx::mbar_arrive(&slot_empty[slot]);
                      }
                    } else {
                      if (lead) ptx::mbar_arrive_expect_tx(&slot_full[slot], C::TILE_BYTES);
                      // the copies start after the lead lane has announced the bytes
                      __syncwarp();
                      uint8_t* dst = smem + C::OFF_RING + slot * C::TILE_BYTES;
                      const int bh_t = t ? w.bh_b : w.bh;
                      const int b = bh_t / h_q;
                      const int kvh = bh_t - b * h_q;
                      const int i = lane * rows;
                      const int key = (w.j0 + j) * kBN + i;
                      if (i < kBN) {
                        int pg = 0;  // rows past the length: page 0, masked later
                        if (key < (t ? w.tkv_b : w.tkv)) {
                          if (staged) {
                            pg = tbl[t * kTblEntries + (key >> pkv.page_shift) - p_lo[t]];
                          } else {
                            pg = __ldg(pkv.table + static_cast<size_t>(b) * pkv.max_pages +
                                       (key >> pkv.page_shift));
                            if (static_cast<unsigned>(pg) >= static_cast<unsigned>(pkv.num_pages)) {
                              atomicCAS(status, 0u,
                                        status_word_code(1u /* ATTN_ERR_INVALID_ARG */,
                                                         kKernPrefill, kSiteBadPage));
                              pg = 0;
                            }
                          }
                        }
                        ptx::tma_load_3d(dst + i * 128, kind ? &tmV : &tmK, &slot_full[slot], 0,
                                         key & ((1 << pkv.page_shift) - 1), pg * h_q + kvh, pol_kv);
                      }
                      // the stand-in release for the other tile
                      if (lead) ptx::mbar_arrive(&slot_empty[slot]);
                    }
                    ++g;
                  }
                }
              }
              // every lane is done with the staged entries before the next
              // unit overwrites them
              __syncwarp();
              continue;
            }
            for (int j = 0; ok && j < w.n_all; ++j) {
              for (int kind = 0; ok && kind < 2; ++kind) {
                for (int t = 0; ok && t < nt; ++t) {
                  const uint32_t slot = g % SL;
                  ok = ptx::mbar_wait(&slot_empty[slot], ((g / SL) & 1) ^ 1, status,
                                      status_word(kKernPrefill, kSiteProdSlot));
                  if (!ok) break;
                  const bool skip = j >= (t ? w.n_b : w.n_a);
                  if (skip) {
                    ptx::mbar_arrive(&slot_full[slot]);
                    ptx::mbar_arrive(&slot_empty[slot]);
                  } else {
                    ptx::mbar_arrive_expect_tx(&slot_full[slot], C::TILE_BYTES);
                    uint8_t* dst = smem + C::OFF_RING + slot * C::TILE_BYTES;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                      ptx::tma_load_3d(dst + c * kSub, kind ? &tmV : &tmK, &slot_full[slot],
                                       c * 64, (w.j0 + j) * kBN, t ? w.kvbh_b : w.kvbh, pol_kv);
                  }
                  ptx::mbar_arrive(&slot_empty[slot]);
                  ++g;
                }
              }
            }
          }
        }
        if (!ok && lead) {
          // Error path: let the copies in flight land before the CTA (and its
          // shared memory) goes away. Only the last SLOTS fills and the last
          // Q load can still be outstanding.
          if (nq > 0) mbar_drain(q_full, (nq - 1) & 1);
          for (uint32_t i = (g > SL ? g - SL : 0); i < g; ++i)
            mbar_drain(&slot_full[i % SL], (i / SL) & 1);
        }
      }
    } else if (warp == kWarpMma || (C::SEP_P && warp == kWarpMma + 1)) {
      // ------------------------------------------------------------ MMA issuer(s)
      // d = 64: warp 9 issues tile A's products and warp 10 tile B's, each in
      // the order its own barriers allow; shared K/V slots and the Q buffer
      // are released by a commit from each. d = 128: warp 9 issues both.
      const int xi = warp - kWarpMma;
      // The whole warp runs this loop in uniform control flow, so descriptor
      // arithmetic stays warp-uniform; one elected lane (the lowest active
      // one, the same every time) issues each batch of MMAs and every commit,
      // so each commit covers that lane's earlier MMAs.
      constexpr uint32_t idS = ptx::make_idesc_f16(BF16, kBM, kBN, false, false);
      constexpr uint32_t idO = ptx::make_idesc_f16(BF16, kBM, D, false, true);
      const uint32_t sQ = ptx::smem_u32(smem + C::OFF_Q);
      const uint32_t sRing = ptx::smem_u32(smem + C::OFF_RING);
      uint32_t g = 0, nq = 0;
      uint32_t np0 = 0, np1 = 0, noe0 = 0, noe1 = 0;
      bool ok = true;

      auto wait_bar = [&](uint64_t* bar, uint32_t parity, uint32_t site) {
        const bool good = ptx::mbar_wait(bar, parity, status, status_word(kKernPrefill, site));
        return __all_sync(0xffffffffu, good);
      };
      auto commit = [&](uint64_t* bar) {
        if (ptx::elect_one_sync()) ptx::mma_commit(bar);
        __syncwarp();
      };
      auto wait_slot = [&](uint32_t idx) {
        return wait_bar(&slot_full[idx % SL], (idx / SL) & 1, kSiteMmaSlot);
      };
      const uint64_t desc_q0 = ptx::make_sdesc_sw128(sQ, 16, 1024);
      const uint64_t desc_k0 = ptx::make_sdesc_sw128(sRing, 16, 1024);
      const uint64_t desc_v0 = ptx::make_sdesc_sw128(sRing, kSub, 1024);
      auto issue_s = [&](int x, uint32_t kslot) {
        const uint64_t qd = desc_q0 + ((x * C::TILE_BYTES) >> 4);
        const uint64_t kd = desc_k0 + ((kslot * C::TILE_BYTES) >> 4);
        const uint32_t d_s = tmem + col_s(x);
        if (ptx::elect_one_sync()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kSub + (kk & 3) * 32;
            ptx::mma_f16_ss(d_s, qd + (koff >> 4), kd + (koff >> 4), idS, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&s_full[x]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int x, uint32_t vslot, bool first) {
        const uint64_t vd = desc_v0 + ((vslot * C::TILE_BYTES) >> 4);
        const uint32_t d_o = tmem + col_o<D>(x);
        const uint32_t a_p = tmem + col_s(x);
        const uint32_t acc0 = first ? 0u : 1u;
        if (ptx::elect_one_sync()) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            ptx::mma_f16_ts(d_o, a_p + kk * 8, vd + ((kk * 16 * 128) >> 4), idO,
                            kk > 0 ? 1u : acc0);
        }
        __syncwarp();
      };
      auto wait_p = [&](int x, bool first) {
        // (scalar counters per tile: an array indexed by the tile would live
        // in local memory)
        bool good = wait_bar(&p_full[x], (x ? np1 : np0) & 1, kSiteMmaP);
        if (x) ++np1; else ++np0;
        if (good && first) {
          // O_X is overwritten by this unit's first product: the previous
          // unit's epilogue must have read it.
          good = wait_bar(&o_empty[x], ((x ? noe1 : noe0) & 1) ^ 1, kSiteMmaOEmpty);
          if (x) ++noe1; else ++noe0;
        }
        ptx::tc_fence_after();
        return good;
      };

      if constexpr (C::SEP_P) {
        // S_X(t) may overwrite S_X once the softmax has read S_X(t-1)
        uint32_t ns_iss = 0;  // score products this warp issued (its tile only)
        auto issue_s_sep = [&](int x, uint32_t kslot) {
          if (ns_iss > 0 && !wait_bar(&s_free[x], (ns_iss - 1) & 1, kSiteMmaSFree)) return false;
          ptx::tc_fence_after();
          issue_s(x, kslot);
          ++ns_iss;
          return true;
        };
        auto issue_pv_sep = [&](int x, uint32_t vslot, bool first) {
          const uint64_t vd = desc_v0 + ((vslot * C::TILE_BYTES) >> 4);
          const uint32_t d_o = tmem + col_o<D>(x);
          const uint32_t a_p = tmem + col_p(x);
          const uint32_t acc0 = first ? 0u : 1u;
          if (ptx::elect_one_sync()) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              ptx::mma_f16_ts(d_o, a_p + kk * 8, vd + ((kk * 16 * 128) >> 4), idO,
                              kk > 0 ? 1u : acc0);
            ptx::mma_commit(&pv_done[x]);
          }
          __syncwarp();
        };
        const int x = xi;  // this warp's tile
        for (int r = 0; ok && r * G < U; ++r) {
          const int u = unit_of_round(r, bid, G);
          if (u >= U) continue;
          const Unit w = unit_info<HP>(u, BH, n_pairs, T_q, T_kv, causal, h_q, h_kv, S, pkv.lens);
          if (w.n_all == 0) continue;  // skipped by the producer too
          const int n_x = x ? w.n_b : w.n_a;
          ok = wait_bar(q_full, nq & 1, kSiteMmaQ);
          ++nq;
          if (!ok) break;
          if constexpr (HP) {
            // this tile's own slots: per key tile the ring holds K_A, K_B,
            // V_A, V_B (K_A, V_A when there is no tile B); the producer
            // stands in for the other tile's releases and for key tiles this
            // tile does not see
            const uint32_t per = w.rows_b > 0 ? 4u : 2u;
            const uint32_t kx = g + static_cast<uint32_t>(x);         // K_0 of this tile
            const uint32_t vx = kx + per / 2;                         // V_0 of this tile
            if (n_x == 0) {
              commit(q_empty);  // no score product of this tile reads Q
            } else {
              ok = wait_slot(kx);
              if (!ok) break;
              ptx::tc_fence_after();
              ok = issue_s_sep(x, kx % SL);
              if (!ok) break;
              commit(&slot_empty[kx % SL]);
              if (n_x == 1) commit(q_empty);
            }
            for (int j = 0; j < n_x; ++j) {
              const uint32_t vi = vx + per * j;        // V_j
              const uint32_t ki = kx + per * (j + 1);  // K_{j+1}
              if (j + 1 < n_x) {
                ok = wait_slot(ki);
                if (!ok) break;
                ptx::tc_fence_after();
                ok = issue_s_sep(x, ki % SL);
                if (!ok) break;
                commit(&slot_empty[ki % SL]);
                if (j + 2 == n_x) commit(q_empty);
              }
              ok = wait_slot(vi);
              if (!ok) break;
              ok = wait_p(x, j == 0);
              if (!ok) break;
              issue_pv_sep(x, vi % SL, j == 0);
              if (j == n_x - 1) commit(&o_full[x]);
              commit(&slot_empty[vi % SL]);
            }
            g += per * w.n_all;
            continue;
          }
          ok = wait_slot(g);  // K_0
          if (!ok) break;
          ptx::tc_fence_after();
          if (n_x > 0) ok = issue_s_sep(x, g % SL);
          if (!ok) break;
          commit(&slot_empty[g % SL]);
          if (n_x <= 1) commit(q_empty);  // no further score product of this tile reads Q
          for (int j = 0; j < w.n_all; ++j) {
            const uint32_t vi = g + 2 * j + 1;  // V_j
            const uint32_t ki = vi + 1;         // K_{j+1}
            if (j + 1 < w.n_all) {
              // scores of the next key tile first: they only need the
              // softmax to have read this tile's scores
              ok = wait_slot(ki);
              if (!ok) break;
              ptx::tc_fence_after();
              if (j + 1 < n_x) ok = issue_s_sep(x, ki % SL);
              if (!ok) break;
              commit(&slot_empty[ki % SL]);
              if (j + 2 == n_x) commit(q_empty);
            }
            ok = wait_slot(vi);
            if (!ok) break;
            if (j < n_x) {
              ok = wait_p(x, j == 0);
              if (!ok) break;
              issue_pv_sep(x, vi % SL, j == 0);
              if (j == n_x - 1) commit(&o_full[x]);
            }
            commit(&slot_empty[vi % SL]);
          }
          g += 2 * w.n_all;
        }
      } else {
        for (int r = 0; ok && r * G < U; ++r) {
          const int u = unit_of_round(r, bid, G);
          if (u >= U) continue;
          const Unit w = unit_info<HP>(u, BH, n_pairs, T_q, T_kv, causal, h_q, h_kv, S, pkv.lens);
          if (w.n_all == 0) continue;  // skipped by the producer too
          ok = wait_bar(q_full, nq & 1, kSiteMmaQ);
          ++nq;
          if (!ok) break;
          // prologue: both score tiles of key tile 0
          ok = wait_slot(g);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s(0, g % SL);
          if (w.n_b > 0) issue_s(1, g % SL);
          commit(&slot_empty[g % SL]);
          if (w.n_all == 1) commit(q_empty);
          for (int j = 0; j < w.n_all; ++j) {
            const uint32_t vi = g + 2 * j + 1;  // V_j
            const uint32_t ki = vi + 1;         // K_{j+1}
            ok = wait_slot(vi);
            if (!ok) break;
            if (j < w.n_a) {
              ok = wait_p(0, j == 0);
              if (!ok) break;
              issue_pv(0, vi % SL, j == 0);
              if (j == w.n_a - 1) commit(&o_full[0]);
            }
            if (j + 1 < w.n_all) {
              ok = wait_slot(ki);
              if (!ok) break;
              ptx::tc_fence_after();
              if (j + 1 < w.n_a) issue_s(0, ki % SL);
            }
            if (j < w.n_b) {
              ok = wait_p(1, j == 0);
              if (!ok) break;
              issue_pv(1, vi % SL, j == 0);
              if (j == w.n_b - 1) commit(&o_full[1]);
            }
            commit(&slot_empty[vi % SL]);
            if (j + 1 < w.n_all) {
              if (j + 1 < w.n_b) issue_s(1, ki % SL);
              commit(&slot_empty[ki % SL]);
              if (j + 2 == w.n_all) commit(q_empty);
            }
          }
          g += 2 * w.n_all;
        }
      }
      // All MMAs this warp issued must be complete before TMEM is freed.
      commit(mma_done);
      mbar_drain(mma_done, 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;                   // 0 = tile A, 1 = tile B
    const int quarter = warp & 3;              // TMEM lanes [32*quarter, 32*quarter+32)
    const int r = quarter * 32 + lane;         // row within the tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t t_s = t_lane + col_s(x);
    const uint32_t t_o = t_lane + col_o<D>(x);
    // where P_X goes: its own columns (SEP_P) or over S_X
    const uint32_t t_p = C::SEP_P ? t_lane + col_p(x) : t_s;
    uint32_t ns = 0, no = 0;
    uint32_t nps = 0;  // P_X tiles stored so far (SEP_P: PV_X(nps - 1) must finish first)
    bool ok = true;

    for (int rr = 0; ok && rr * G < U; ++rr) {
      const int u = unit_of_round(rr, bid, G);
      if (u >= U) continue;
      const Unit w = unit_info<HP>(u, BH, n_pairs, T_q, T_kv, causal, h_q, h_kv, S, pkv.lens);
      const int n_x = x ? w.n_b : w.n_a;
      const int bh_x = HP && x ? w.bh_b : w.bh;      // this tile's head
      const int row = (HP ? 0 : w.q0 + x * kBM) + r;  // absolute query row
      if (n_x == 0) {
        // no key of this partition for this tile: an empty partial (weight 0
        // in the merge) for each of its rows; unsplit (a sequence of length 0
        // in the paged mode), the output of a row with no keys: o = 0,
        // lse = -inf
        if (row < T_q && (x == 0 || w.rows_b > 0)) {
          if (S > 1) {
            float* pr = part + ((static_cast<size_t>(bh_x) * T_q + row) * S + w.s) * (D + 4);
#pragma unroll
            for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(pr + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(pr + D) = make_float4(-INFINITY, 0.f, 0.f, 0.f);
          } else if constexpr (PAGED) {
            // (only a paged sequence can have no keys at all)
            uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(out) +
                                                   (static_cast<size_t>(bh_x) * T_q + row) * D * 2);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0u, 0u, 0u, 0u);
            lse[static_cast<size_t>(bh_x) * T_q + row] = -INFINITY;
          }
        }
        continue;
      }
      const int tkv_x = HP && x ? w.tkv_b : w.tkv;
      const int last_key = causal ? min(tkv_x - 1, row + off) : tkv_x - 1;
      float m_used = -INFINITY;  // reference max, log2 units of the scaled score
      float l = 0.f;

      for (int j = 0; j < n_x; ++j) {
        ok = ptx::mbar_wait(&s_full[x], ns & 1, status, status_word(kKernPrefill, kSiteSoftS));
        ++ns;
        // tcgen05.ld/st/wait are warp-collective (.sync.aligned): every
        // branch around them must be taken by the whole warp.
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[128];
        tmem_ld_row128(t_s, sr);
        if constexpr (C::SEP_P) {
          // the scores are in registers: S_X may be overwritten
          ptx::tc_fence_before();
          ptx::mbar_arrive(&s_free[x]);
        }
        float* s = reinterpret_cast<float*>(sr);

        const int key0 = (w.j0 + j) * kBN;
        if (key0 + kBN - 1 > last_key) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (key0 + c > last_key) s[c] = -INFINITY;
        }
        // row max: four independent chains of 3-input max
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kBN; c += 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) m4[i] = fmax3(m4[i], s[c + 2 * i], s[c + 2 * i + 1]);
        }
        const float mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        const float m_tile = mx * scale_log2;
        float alpha = 1.f;
        bool rescale = false;
        if (m_tile > m_used + kRebaseLog2) {
          alpha = ptx::ex2_approx(m_used - m_tile);  // 0 when m_used = -inf
          rescale = (m_used != -INFINITY);
          l *= alpha;
          m_used = m_tile;
        }
        const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;

        // p = 2^(s * scale * log2e - m_ref), two columns per instruction
        const float2 sl2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_ref, -m_ref);
        float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};  // four independent sum chains
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          const float2 xx = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2, nm2);
          float2 pp;
          pp.x = ptx::ex2_approx(xx.x);
          pp.y = ptx::ex2_approx(xx.y);
          rs2[(c >> 1) & 3] = __fadd2_rn(rs2[(c >> 1) & 3], pp);
          pk[c >> 1] = pack2<BF16>(pp.x, pp.y);
        }
        const float2 rsa = __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
        l += rsa.x + rsa.y;
        // the exponentials are done here, not after the wait for PV_X below
        reg_fence64f(pk, l);

        if constexpr (C::SEP_P) {
          // P_X and O_X are free once the previous product PV_X finished
          if (nps > 0) {
            ok = ptx::mbar_wait(&pv_done[x], (nps - 1) & 1, status,
                                status_word(kKernPrefill, kSiteSoftPv));
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
          }
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // O_X holds the sum through key tile j-1 (that product is complete:
          // without SEP_P it was issued before S_X(j), whose completion this
          // warp waited for; with SEP_P this warp waited for it just above).
          // Multiply this warp's rows by their alpha in place; rows that keep
          // their reference max multiply by 1.
          const float mul = rescale ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t raw[32];
            ptx::tmem_ld_32x32b_x32(t_o + c * 32, raw);
            tmem_wait_ld_regs(raw);
#pragma unroll
            for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * mul);
            ptx::tmem_st_32x32b_x32(t_o + c * 32, raw);
          }
        }
        // P_X (16-bit pairs) into its columns (or the first 64 of S_X)
        ptx::tmem_st_32x32b_x32(t_p, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        ptx::tmem_st_32x32b_x32(t_p + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&p_full[x]);
        ++nps;
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      ok = ptx::mbar_wait(&o_full[x], no & 1, status, status_word(kKernPrefill, kSiteSoftO));
      ++no;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const bool write = row < T_q;
      if (S > 1) {
        // partial of key partition s: unnormalised o, and (m, l) in log2
        // units of the scaled score -- the decode partial format
        float* pr = part + ((static_cast<size_t>(bh_x) * T_q + (write ? row : 0)) * S + w.s) * (D + 4);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t raw[32];
          ptx::tmem_ld_32x32b_x32(t_o + c * 32, raw);
          tmem_wait_ld_regs(raw);
          if (write) {
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4)
              *reinterpret_cast<float4*>(pr + c * 32 + g4 * 4) =
                  make_float4(__uint_as_float(raw[4 * g4]), __uint_as_float(raw[4 * g4 + 1]),
                              __uint_as_float(raw[4 * g4 + 2]), __uint_as_float(raw[4 * g4 + 3]));
          }
        }
        if (write) *reinterpret_cast<float4*>(pr + D) = make_float4(m_used, l, 0.f, 0.f);
        ptx::tc_fence_before();
        ptx::mbar_arrive(&o_empty[x]);
        continue;
      }
      const float inv_l = 1.f / l;
      uint8_t* orow = reinterpret_cast<uint8_t*>(out) +
                      (static_cast<size_t>(bh_x) * T_q + (write ? row : 0)) * D * 2;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t raw[32];
        ptx::tmem_ld_32x32b_x32(t_o + c * 32, raw);
        tmem_wait_ld_regs(raw);
        if (write) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            uint4 v;
            const float* f = reinterpret_cast<const float*>(&raw[g8 * 8]);
            v.x = pack2<BF16>(f[0] * inv_l, f[1] * inv_l);
            v.y = pack2<BF16>(f[2] * inv_l, f[3] * inv_l);
            v.z = pack2<BF16>(f[4] * inv_l, f[5] * inv_l);
            v.w = pack2<BF16>(f[6] * inv_l, f[7] * inv_l);
            // O is not read again by this kernel: a streaming store (evict
            // first in L2) leaves the K/V tiles later units re-read in L2
            __stcs(reinterpret_cast<uint4*>(orow + (c * 32 + g8 * 8) * 2), v);
          }
        }
      }
      if (write)
        lse[static_cast<size_t>(bh_x) * T_q + row] = (m_used + __log2f(l)) * 0.69314718055994531f;
      ptx::tc_fence_before();
      ptx::mbar_arrive(&o_empty[x]);
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
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
template <int D, bool BF16, bool PAGED, bool HP>
cudaError_t launch_t(const FwdProblem& p, int S, float* part, cudaStream_t stream,
                     const PagedKV& pkv, const void* k_pool, const void* v_pool) {
  using C = Cfg<D>;
  auto kern = prefill_kernel<D, BF16, PAGED, HP>;
  constexpr int smem_bytes = C::SMEM_BYTES + ((PAGED && HP) ? kTblBytes : 0);
  static std::mutex mu;
  static uint64_t configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64 && !(configured & (1ull << dev))) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
      if (e != cudaSuccess) return e;
      configured |= 1ull << dev;
    }
  }
  const int BH = p.B * p.h;
  CUtensorMap mq, mk, mv;
  const int BH_kv = p.B * p.h_kv;
  if (!make_map(&mq, p.q, p.T_q, BH, D, BF16, kBM)) return cudaErrorInvalidValue;
  if constexpr (PAGED) {
    // the pool as [num_pages * h_kv][page_size][D], boxes of min(page_size, 128) rows
    const int ps = 1 << pkv.page_shift;
    if (!make_map(&mk, k_pool, ps, pkv.num_pages * p.h_kv, D, BF16, ps < kBN ? ps : kBN) ||
        !make_map(&mv, v_pool, ps, pkv.num_pages * p.h_kv, D, BF16, ps < kBN ? ps : kBN))
      return cudaErrorInvalidValue;
  } else {
    if (!make_map(&mk, p.k, p.T_kv, BH_kv, D, BF16, kBN) ||
        !make_map(&mv, p.v, p.T_kv, BH_kv, D, BF16, kBN))
      return cudaErrorInvalidValue;
  }
  const int n_qtiles = (p.T_q + kBM - 1) / kBM;
  const int n_pairs = (n_qtiles + 1) / 2;
  const long long units =
      static_cast<long long>(HP ? (BH + 1) / 2 : static_cast<long long>(n_pairs) * BH) * S;
  const int sms = device_sms(dev);
  const int grid = static_cast<int>(units < sms ? units : sms);
  const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
  kern<<<grid, kThreads, smem_bytes, stream>>>(mq, mk, mv, p.o, p.lse, p.T_q, p.T_kv, BH, n_pairs,
                                                  scale_log2, p.causal, p.status, p.h, p.h_kv, S,
                                                  part, pkv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const FwdProblem& p, int num_splits, float* part, cudaStream_t stream,
                           const char** name) {
  cudaError_t e;
  const bool split = num_splits > 1;
  const PagedKV none{nullptr, nullptr, 0, 0, 0};
  if (p.d == 64) {
    // short queries: two heads per unit (head-pair mode)
    if (head_pair_mode(64, p.T_q, static_cast<long long>(p.B) * p.h))
      e = p.bf16 ? launch_t<64, true, false, true>(p, num_splits, part, stream, none, nullptr, nullptr)
                 : launch_t<64, false, false, true>(p, num_splits, part, stream, none, nullptr, nullptr);
    else
      e = p.bf16 ? launch_t<64, true, false, false>(p, num_splits, part, stream, none, nullptr, nullptr)
                 : launch_t<64, false, false, false>(p, num_splits, part, stream, none, nullptr, nullptr);
    *name = split ? (p.bf16 ? "prefill_splitkv_tcgen05_d64_bf16+decode_combine"
                            : "prefill_splitkv_tcgen05_d64_f16+decode_combine")
                  : (p.bf16 ? "prefill_tcgen05_d64_bf16" : "prefill_tcgen05_d64_f16");
  } else {
    e = p.bf16 ? launch_t<128, true, false, false>(p, num_splits, part, stream, none, nullptr, nullptr)
               : launch_t<128, false, false, false>(p, num_splits, part, stream, none, nullptr, nullptr);
    *name = split ? (p.bf16 ? "prefill_splitkv_tcgen05_d128_bf16+decode_combine"
                            : "prefill_splitkv_tcgen05_d128_f16+decode_combine")
                  : (p.bf16 ? "prefill_tcgen05_d128_bf16" : "prefill_tcgen05_d128_f16");
  }
  if (e != cudaSuccess || !split) return e;
  // merge the partials of each query row: rows = B*h*T_q
  return launch_combine(part, p.o, p.lse, static_cast<long long>(p.B) * p.h * p.T_q, num_splits,
                        p.d, p.bf16 != 0, stream);
}

}  // namespace attn

namespace attn {

cudaError_t launch_prefill_paged(const FwdProblem& p, const int* table, const int* lens,
                                 int page_shift, int max_pages, int num_pages, int num_splits,
                                 float* part, cudaStream_t stream, const char** name) {
  const PagedKV pkv{table, lens, page_shift, max_pages, num_pages};
  cudaError_t e;
  if (p.d == 64) {
    // two heads per unit (head pairs) when the query rows fit one tile and
    // the pages hold 64 rows or more
    if (paged_head_pairs(64, p.T_q, static_cast<long long>(p.B) * p.h, 1 << page_shift))
      e = p.bf16 ? launch_t<64, true, true, true>(p, num_splits, part, stream, pkv, p.k, p.v)
                 : launch_t<64, false, true, true>(p, num_splits, part, stream, pkv, p.k, p.v);
    else
      e = p.bf16 ? launch_t<64, true, true, false>(p, num_splits, part, stream, pkv, p.k, p.v)
                 : launch_t<64, false, true, false>(p, num_splits, part, stream, pkv, p.k, p.v);
    *name = p.bf16 ? "prefill_paged_tcgen05_d64_bf16+decode_combine"
                   : "prefill_paged_tcgen05_d64_f16+decode_combine";
  } else {
    e = p.bf16 ? launch_t<128, true, true, false>(p, num_splits, part, stream, pkv, p.k, p.v)
               : launch_t<128, false, true, false>(p, num_splits, part, stream, pkv, p.k, p.v);
    *name = p.bf16 ? "prefill_paged_tcgen05_d128_bf16+decode_combine"
                   : "prefill_paged_tcgen05_d128_f16+decode_combine";
  }
  if (e != cudaSuccess) return e;
  if (num_splits <= 1) return cudaSuccess;  // the kernel wrote o and lse
  return launch_combine(part, p.o, p.lse, static_cast<long long>(p.B) * p.h * p.T_q, num_splits,
                        p.d, p.bf16 != 0, stream);
}

}  // namespace attn
