// attn_api.cu -- the C ABI of libattn (declared in include/attn.h): argument
// validation; dispatch of prefill, decode (CUDA cores, or the tensor cores
// for grouped-query groups of 4 or more), paged decode, split-KV prefill and
// backward; the split-count choices; stream-ordered workspace; the
// host-buffer entry's copies; and the device status word. All compute happens
// in the kernels of prefill_sm103.cu, decode_sm103.cu and backward_sm103.cu;
// nothing here computes attention.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"
#include "attn_status.h"
#include "ptx_sm103.cuh"

namespace {

// One status word per device (each device's module instance has its own).
__device__ unsigned int g_status_word;

// Failure-detection self-test: one thread waits on an mbarrier that nothing
// will ever complete, with the same bounded wait the attention kernels use
// but a short limit. The wait gives up, records the timeout in the status
// word and the kernel returns; nothing faults or hangs.
__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    attn::ptx::mbar_init(&bar, 1);
    attn::ptx::fence_mbarrier_init();
    attn::ptx::mbar_wait_for(&bar, 0, status, attn::status_word(attn::kKernSelftest, 1), limit_ns);
  }
}

unsigned int* status_ptr() {
  static std::mutex mu;
  static unsigned int* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

int sm_count() {
  static std::mutex mu;
  static int counts[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> g(mu);
  if (!counts[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    counts[dev] = n;
  }
  return counts[dev];
}

int split_ctas_per_sm(int d, int heads_per_cta) {
  static std::mutex mu;
  static int cache[64][2][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  const int gi = heads_per_cta >= 8 ? 3 : heads_per_cta >= 4 ? 2 : heads_per_cta >= 2 ? 1 : 0;
  std::lock_guard<std::mutex> g(mu);
  int& c = cache[dev][d == 128][gi];
  if (!c) c = attn::decode_split_ctas_per_sm(d, heads_per_cta);
  return c;
}

thread_local const char* t_last_kernel = "none";

constexpr int kMaxSplits = 1024;

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace attn {
namespace detail {

// Validates everything that does not depend on the workspace. Sets *empty
// when the output has no elements (a valid no-op).
attn_status_t validate(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int h, int T_q, int T_kv, int d, float scale, int causal, int dtype,
                       bool* empty, int h_kv) {
  *empty = false;
  if (h_kv < 0) h_kv = h;  // plain attention: one key/value head per query head
  if (B < 0 || h < 0 || T_q < 0 || T_kv < 0) return ATTN_ERR_INVALID_ARG;
  if (h > 0 && (h_kv < 1 || h % h_kv != 0)) return ATTN_ERR_INVALID_ARG;
  if (d <= 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * h;
  if (BH >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  if (BH == 0 || T_q == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (T_kv < 1) return ATTN_ERR_INVALID_ARG;
  if (causal && T_q > T_kv) return ATTN_ERR_INVALID_ARG;
  if (T_q > 1) {
    // prefill grid: one CTA per (query tile of 128 rows, b, h)
    const long long tiles = (static_cast<long long>(T_q) + 127) / 128;
    if (tiles * BH > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  }
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  const size_t qo_bytes = static_cast<size_t>(BH) * T_q * d * 2;
  const size_t kv_bytes = static_cast<size_t>(B) * h_kv * T_kv * d * 2;
  const size_t lse_bytes = static_cast<size_t>(BH) * T_q * 4;
  if (overlaps(o, qo_bytes, q, qo_bytes) || overlaps(o, qo_bytes, k, kv_bytes) ||
      overlaps(o, qo_bytes, v, kv_bytes) || overlaps(o, qo_bytes, lse, lse_bytes) ||
      overlaps(lse, lse_bytes, q, qo_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
      overlaps(lse, lse_bytes, v, kv_bytes))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Decode split count chosen by shape. The split kernel streams the cache at
// the HBM rate once the device holds enough CTAs, and CTAs that start late
// (the last, partly filled wave) cost time in proportion to their share of a
// wave. So: aim at about eight waves of CTAs (rows * S ~ 8 * cap, cap = SMs x
// resident CTAs per SM), then, within a quarter either side of that count,
// take the S whose last wave is fullest, the smallest such S on ties (less
// merge work). Partitions keep at least 128 keys each. Measured on the
// 32 x 12-head, 16K-key decode: 6 to 10 waves all run within 2% of each other
// and of the bandwidth bound; a last wave a few percent full costs ~10%.
// `rows` = split CTAs per partition index (B * h for plain attention).
int choose_splits(long long rows, int T_kv, int d, int heads_per_cta) {
  return choose_splits_cap(rows, T_kv,
                           static_cast<long long>(sm_count()) * split_ctas_per_sm(d, heads_per_cta));
}

int choose_splits_cap(long long rows, int T_kv, long long cap) {
  const long long max_s = std::max(1ll, std::min<long long>(kMaxSplits, T_kv / 128));
  const long long target = std::min(max_s, std::max(1ll, (8 * cap + rows / 2) / rows));
  const long long lo = std::max(1ll, (target * 3) / 4);
  const long long hi = std::min(max_s, (target * 5 + 3) / 4);
  long long best = lo;
  double best_fill = -1.0;
  for (long long s = lo; s <= hi; ++s) {
    const long long ctas = rows * s;
    const long long waves = (ctas + cap - 1) / cap;
    const double fill = static_cast<double>(ctas) / static_cast<double>(waves * cap);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = s;
    }
  }
  return static_cast<int>(best);
}

}  // namespace detail
}  // namespace attn

namespace {

using attn::detail::choose_splits;
using attn::detail::validate;

size_t ws_bytes(int B, int h, int d, int splits) {
  return static_cast<size_t>(B) * h * splits * attn::decode_partial_floats(d) * sizeof(float);
}

// Split CTAs per partition index of a decode call.
long long decode_rows(int B, int h, int h_kv) {
  const int g = h / h_kv;
  return static_cast<long long>(B) * h_kv * (g / attn::decode_heads_per_cta(g));
}

// Grouped-query decode with at least this many query heads per key/value
// head runs on the tensor cores: the group's query rows are contiguous in q
// ([B][h_q][1][d] is [B][h_kv][G][d]), so the decode is a non-causal prefill
// of T_q = G rows per key/value head, cut into key partitions and merged
// exactly (the split-KV prefill). The CUDA-core split kernel does
// 2*d*G FMAs per cached key and runs out of issue slots at large G.
constexpr int kTensorGroup = 4;
bool gqa_decode_on_tensor_cores(int h, int h_kv) { return h_kv > 0 && h / h_kv >= kTensorGroup; }
// Paged decode with groups of kTensorGroup or more and pages of at least 8
// rows (whole 1024-byte swizzle atoms per TMA box) runs on the tensor cores:
// the prefill kernel gathering K/V tiles through the block table.
bool paged_on_tensor_cores(int h_q, int h_kv, int page_size) {
  return gqa_decode_on_tensor_cores(h_q, h_kv) && page_size >= 8;
}

// Tensor-core forward units per key partition and query-tile pair: B*h
// heads, or head pairs in head-pair mode (attn_internal.h).
long long tc_units(int B, int h, int T_q, int d) {
  const long long bh = static_cast<long long>(B) * h;
  return attn::head_pair_mode(d, T_q, bh) ? (bh + 1) / 2 : bh;
}

int auto_splits(int B, int h, int h_kv, int T_kv, int d) {
  if (gqa_decode_on_tensor_cores(h, h_kv))  // one prefill CTA per SM, per unit of heads
    return std::min(64, attn::detail::choose_splits_cap(tc_units(B, h_kv, h / h_kv, d), T_kv,
                                                        sm_count()));
  return choose_splits(decode_rows(B, h, h_kv), T_kv, d, attn::decode_heads_per_cta(h / h_kv));
}

// Prefill key partitions: only when the (query-tile pair, head) units fill
// less than half the SMs; then enough partitions to reach about one unit per
// SM, at least 2 key tiles each, at most 64.
int prefill_auto_splits(int B, int h, int T_q, int T_kv, int d) {
  const long long pairs = ((static_cast<long long>(T_q) + 127) / 128 + 1) / 2;
  const long long units = tc_units(B, h, T_q, d) * pairs;
  const long long sms = sm_count();
  if (units * 2 > sms) return 1;
  const long long n_kv = (static_cast<long long>(T_kv) + 127) / 128;
  const long long s = std::min({(sms + units - 1) / units, n_kv / 2, 64ll});
  return static_cast<int>(std::max(1ll, s));
}

size_t prefill_ws_bytes(int B, int h, int T_q, int d, int splits) {
  return splits > 1 ? static_cast<size_t>(B) * h * T_q * splits * attn::decode_partial_floats(d) *
                          sizeof(float)
                    : 0;
}

// Prefill with `splits` key partitions (1: the plain kernel, no workspace).
// Every argument check comes before the first CUDA call.
attn_status_t run_prefill(attn::FwdProblem p, int splits, void* workspace, size_t workspace_bytes,
                          bool own, cudaStream_t s) {
  const char* name = "none";
  if (splits <= 1) {
    p.status = status_ptr();
    if (!p.status) return ATTN_ERR_CUDA;
    if (attn::launch_prefill(p, 1, nullptr, s, &name) != cudaSuccess) return ATTN_ERR_CUDA;
    t_last_kernel = name;
    return ATTN_OK;
  }
  const long long rows = static_cast<long long>(p.B) * p.h * p.T_q;
  const long long pairs = ((static_cast<long long>(p.T_q) + 127) / 128 + 1) / 2;
  if (rows > 0x7fffffffll || pairs * p.B * p.h * splits > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  const size_t need = prefill_ws_bytes(p.B, p.h, p.T_q, p.d, splits);
  float* ws = static_cast<float*>(workspace);
  if (!own) {
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return ATTN_ERR_WORKSPACE;
    const size_t qo = static_cast<size_t>(rows) * p.d * 2;
    const size_t kv = static_cast<size_t>(p.B) * p.h_kv * p.T_kv * p.d * 2;
    if (overlaps(workspace, need, p.q, qo) || overlaps(workspace, need, p.k, kv) ||
        overlaps(workspace, need, p.v, kv) || overlaps(workspace, need, p.o, qo) ||
        overlaps(workspace, need, p.lse, static_cast<size_t>(rows) * 4))
      return ATTN_ERR_WORKSPACE;
  }
  p.status = status_ptr();
  if (!p.status) return ATTN_ERR_CUDA;
  if (own && cudaMallocAsync(reinterpret_cast<void**>(&ws), need, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const cudaError_t e = attn::launch_prefill(p, splits, ws, s, &name);
  if (own) cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  t_last_kernel = name;
  return ATTN_OK;
}

attn_status_t run(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                  int h_kv, int T_q, int T_kv, int d, float scale, int causal, int dtype,
                  int num_splits, void* workspace, size_t workspace_bytes, bool own_workspace,
                  void* stream) {
  bool empty = false;
  attn_status_t st = validate(q, k, v, o, lse, B, h, T_q, T_kv, d, scale, causal, dtype, &empty,
                              h_kv);
  if (st != ATTN_OK) return st;
  if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  if (empty) {
    t_last_kernel = "none";
    return ATTN_OK;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  attn::FwdProblem p{q, k, v, o, lse, B, h, T_q, T_kv, d, scale, causal, dtype == ATTN_BF16 ? 1 : 0,
                     nullptr, h_kv};
  const char* name = "none";
  if (T_q > 1) {
    // attn_fwd (own workspace) cuts the key range of small problems into
    // partitions; attn_fwd_ex and attn_fwd_gqa with a caller workspace keep
    // the prefill unsplit (their workspace contract is decode-only)
    const int splits = own_workspace ? prefill_auto_splits(B, h, T_q, T_kv, d) : 1;
    return run_prefill(p, splits, nullptr, 0, true, s);
  }
  // the same choice attn_workspace_bytes(..., 0) reports (occupancy of the bf16
  // and fp16 split kernels is identical)
  const int splits = num_splits > 0 ? num_splits : auto_splits(B, h, h_kv, T_kv, d);
  if (gqa_decode_on_tensor_cores(h, h_kv)) {
    // the G = h/h_kv query heads of each key/value head as G query rows
    // of one virtual head: B*h_kv heads, T_q = G, no mask; partials and
    // outputs land in the same [B*h][...] order as the decode's
    if (splits > 64) return ATTN_ERR_UNSUPPORTED;
    attn::FwdProblem g{q, k, v, o, lse, B, h_kv, h / h_kv, T_kv, d, scale, 0,
                       dtype == ATTN_BF16 ? 1 : 0, nullptr, h_kv};
    return run_prefill(g, splits, workspace, workspace_bytes, own_workspace, s);
  }
  // split grid: one CTA per (row of query heads, partition)
  if (decode_rows(B, h, h_kv) * splits > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  const size_t need = ws_bytes(B, h, d, splits);
  if (!own_workspace) {
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return ATTN_ERR_WORKSPACE;
    if (overlaps(workspace, need, q, static_cast<size_t>(B) * h * d * 2) ||
        overlaps(workspace, need, k, static_cast<size_t>(B) * h_kv * T_kv * d * 2) ||
        overlaps(workspace, need, v, static_cast<size_t>(B) * h_kv * T_kv * d * 2) ||
        overlaps(workspace, need, o, static_cast<size_t>(B) * h * d * 2) ||
        overlaps(workspace, need, lse, static_cast<size_t>(B) * h * 4))
      return ATTN_ERR_WORKSPACE;
  }
  p.status = status_ptr();
  if (!p.status) return ATTN_ERR_CUDA;
  float* ws = static_cast<float*>(workspace);
  if (own_workspace) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&ws), need, s) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  const cudaError_t e = attn::launch_decode(p, splits, ws, s, &name);
  if (own_workspace) cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  t_last_kernel = name;
  return ATTN_OK;
}

// Backward: the forward's checks on (q, k, v, o, lse), then dout, the three
// gradients and the workspace.
attn_status_t run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, int B, int h, int h_kv,
                      int T_q, int T_kv, int d, float scale, int causal, int dtype,
                      void* workspace, size_t workspace_bytes, void* stream) {
  bool empty = false;
  attn_status_t st = validate(q, k, v, const_cast<void*>(o), const_cast<float*>(lse), B, h, T_q,
                              T_kv, d, scale, causal, dtype, &empty, h_kv);
  if (st != ATTN_OK) return st;
  if (empty) {
    t_last_kernel = "none";
    return ATTN_OK;
  }
  const long long BH = static_cast<long long>(B) * h;
  const long long key_tiles = (static_cast<long long>(T_kv) + 127) / 128;
  const long long q_tiles = (static_cast<long long>(T_q) + 127) / 128;
  // grids: one CTA per (key tile, kv head), one per (query tile, head), and
  // the row-term pass at 16 rows per CTA over 128 rows per query tile
  if (key_tiles * B * h_kv > 0x7fffffffll || q_tiles * BH * 8 > 0x7fffffffll)
    return ATTN_ERR_UNSUPPORTED;
  if (!dout || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return ATTN_ERR_INVALID_ARG;
  const size_t qo_bytes = static_cast<size_t>(BH) * T_q * d * 2;
  const size_t kv_bytes = static_cast<size_t>(B) * h_kv * T_kv * d * 2;
  const size_t lse_bytes = static_cast<size_t>(BH) * T_q * 4;
  struct Buf { const void* p; size_t n; };
  const Buf ins[] = {{q, qo_bytes}, {k, kv_bytes}, {v, kv_bytes}, {o, qo_bytes},
                     {dout, qo_bytes}, {lse, lse_bytes}};
  const Buf outs[] = {{dq, qo_bytes}, {dk, kv_bytes}, {dv, kv_bytes}};
  for (int i = 0; i < 3; ++i) {
    for (const Buf& b : ins)
      if (overlaps(outs[i].p, outs[i].n, b.p, b.n)) return ATTN_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return ATTN_ERR_INVALID_ARG;
  }
  const size_t need = attn::bwd_workspace_floats(BH, T_q) * sizeof(float);
  const bool own = workspace == nullptr && workspace_bytes == 0;
  if (!own) {
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return ATTN_ERR_WORKSPACE;
    for (const Buf& b : ins)
      if (overlaps(workspace, need, b.p, b.n)) return ATTN_ERR_WORKSPACE;
    for (const Buf& b : outs)
      if (overlaps(workspace, need, b.p, b.n)) return ATTN_ERR_WORKSPACE;
  }
  attn::BwdProblem p{q, k, v, o, dout, lse, dq, dk, dv, B, h, h_kv, T_q, T_kv, d, scale, causal,
                     dtype == ATTN_BF16 ? 1 : 0, nullptr, status_ptr()};
  if (!p.status) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  if (own) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&ws), need, s) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  p.ws = ws;
  const char* name = "none";
  const cudaError_t e = attn::launch_backward(p, s, &name);
  if (own) cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  t_last_kernel = name;
  return ATTN_OK;
}


int paged_ctas_per_sm(int d) {
  static std::mutex mu;
  static int cache[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  std::lock_guard<std::mutex> g(mu);
  int& c = cache[dev][d == 128];
  if (!c) c = attn::decode_paged_ctas_per_sm(d);
  return c;
}

// Paged decode: the split count for a shape, from the longest cache the
// block table can name (the lengths live on the device).
int paged_auto_splits(int B, int h_q, int h_kv, int d, int page_size, int max_pages) {
  const long long t = std::min<long long>(0x7fffffffll, static_cast<long long>(page_size) * max_pages);
  if (paged_on_tensor_cores(h_q, h_kv, page_size)) {  // one prefill CTA per SM, per unit of heads
    const long long bh = static_cast<long long>(B) * h_kv;
    const long long units =
        attn::paged_head_pairs(d, h_q / h_kv, bh, page_size) ? (bh + 1) / 2 : bh;
    return std::min(64, attn::detail::choose_splits_cap(units, static_cast<int>(t), sm_count()));
  }
  const long long cap = static_cast<long long>(sm_count()) * paged_ctas_per_sm(d);
  return attn::detail::choose_splits_cap(static_cast<long long>(B) * h_q, static_cast<int>(t), cap);
}

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

attn_status_t run_paged(const void* q, const void* k_pages, const void* v_pages,
                        const int* block_table, const int* seq_lens, void* o, float* lse, int B,
                        int h_q, int h_kv, int d, int page_size, int max_pages, int num_pages,
                        float scale, int dtype, int num_splits, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (B < 0 || h_q < 0 || h_kv < 1 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (h_q % h_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!pow2(page_size) || page_size > 65536 || max_pages < 1 || num_pages < 1)
    return ATTN_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(page_size) * max_pages > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * h_q;
  if (BH == 0) {
    t_last_kernel = "none";
    return ATTN_OK;
  }
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !o || !lse)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(o, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  const int splits =
      num_splits > 0 ? num_splits : paged_auto_splits(B, h_q, h_kv, d, page_size, max_pages);
  if (BH * splits > 0x7fffffffll) return ATTN_ERR_UNSUPPORTED;
  const size_t qo = static_cast<size_t>(BH) * d * 2;
  const size_t pool = static_cast<size_t>(num_pages) * h_kv * page_size * d * 2;
  const size_t tab = static_cast<size_t>(B) * max_pages * 4;
  const size_t lens = static_cast<size_t>(B) * 4;
  const size_t lse_b = static_cast<size_t>(BH) * 4;
  struct Buf { const void* p; size_t n; };
  const Buf ins[] = {{q, qo}, {k_pages, pool}, {v_pages, pool}, {block_table, tab}, {seq_lens, lens}};
  for (const Buf& b : ins)
    if (overlaps(o, qo, b.p, b.n) || overlaps(lse, lse_b, b.p, b.n)) return ATTN_ERR_INVALID_ARG;
  if (overlaps(o, qo, lse, lse_b)) return ATTN_ERR_INVALID_ARG;
  // (the tensor-core path with one partition writes o directly: no workspace)
  const bool tc = paged_on_tensor_cores(h_q, h_kv, page_size);
  const size_t need = (tc && splits <= 1) ? 0 : ws_bytes(B, h_q, d, splits);
  const bool own = workspace == nullptr && workspace_bytes == 0;
  if (!own && need > 0) {
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return ATTN_ERR_WORKSPACE;
    for (const Buf& b : ins)
      if (overlaps(workspace, need, b.p, b.n)) return ATTN_ERR_WORKSPACE;
    if (overlaps(workspace, need, o, qo) || overlaps(workspace, need, lse, lse_b))
      return ATTN_ERR_WORKSPACE;
  }
  int shift = 0;
  while ((1 << shift) < page_size) ++shift;
  if (tc) {
    if (splits > 64) return ATTN_ERR_UNSUPPORTED;
    // virtual problem: B*h_kv heads of T_q = G query rows against the pages
    attn::FwdProblem g{q, k_pages, v_pages, o, lse, B, h_kv, h_q / h_kv, page_size * max_pages, d,
                       scale, 0, dtype == ATTN_BF16 ? 1 : 0, status_ptr(), h_kv};
    if (!g.status) return ATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* ws = static_cast<float*>(workspace);
    if (own && splits > 1 &&
        cudaMallocAsync(reinterpret_cast<void**>(&ws), need, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    const char* name = "none";
    const cudaError_t e = attn::launch_prefill_paged(g, block_table, seq_lens, shift, max_pages,
                                                     num_pages, splits, ws, s, &name);
    if (own && splits > 1) cudaFreeAsync(ws, s);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    t_last_kernel = name;
    return ATTN_OK;
  }
  attn::PagedProblem p{q, k_pages, v_pages, block_table, seq_lens, o, lse, B, h_q, h_kv, d, shift,
                       max_pages, num_pages, scale, dtype == ATTN_BF16 ? 1 : 0, status_ptr()};
  if (!p.status) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  if (own) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&ws), need, s) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  const char* name = "none";
  const cudaError_t e = attn::launch_decode_paged(p, splits, ws, s, &name);
  if (own) cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  t_last_kernel = name;
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int h, int T_q, int T_kv, int d, float scale, int causal, int dtype,
                       void* stream) {
  return run(q, k, v, o, lse, B, h, h, T_q, T_kv, d, scale, causal, dtype, 0, nullptr, 0, true,
             stream);
}

attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int h, int T_q, int T_kv, int d, float scale, int causal, int dtype,
                          int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  return run(q, k, v, o, lse, B, h, h, T_q, T_kv, d, scale, causal, dtype, num_splits, workspace,
             workspace_bytes, false, stream);
}

attn_status_t attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                           int causal, int dtype, int num_splits, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (h_kv < 1) return ATTN_ERR_INVALID_ARG;
  const bool own = workspace == nullptr && workspace_bytes == 0;
  return run(q, k, v, o, lse, B, h_q, h_kv, T_q, T_kv, d, scale, causal, dtype, num_splits,
             workspace, workspace_bytes, own, stream);
}

attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                               int causal, int dtype, int num_splits, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (h_kv < 1) return ATTN_ERR_INVALID_ARG;
  bool empty = false;
  attn_status_t st = validate(q, k, v, o, lse, B, h_q, T_q, T_kv, d, scale, causal, dtype, &empty,
                              h_kv);
  if (st != ATTN_OK) return st;
  if (num_splits < 0 || num_splits > 64) return ATTN_ERR_INVALID_ARG;
  if (T_q < 2) return ATTN_ERR_INVALID_ARG;  // one query row: use the decode entries
  if (empty) {
    t_last_kernel = "none";
    return ATTN_OK;
  }
  attn::FwdProblem p{q, k, v, o, lse, B, h_q, T_q, T_kv, d, scale, causal,
                     dtype == ATTN_BF16 ? 1 : 0, nullptr, h_kv};
  const int splits = num_splits > 0 ? num_splits : prefill_auto_splits(B, h_q, T_q, T_kv, d);
  const bool own = workspace == nullptr && workspace_bytes == 0;
  return run_prefill(p, splits, workspace, workspace_bytes, own, static_cast<cudaStream_t>(stream));
}

// Device copies of a host-buffer call: q | k | v | o | lse, each at a
// 256-byte offset. Returns 0 for shapes the forward rejects or an empty one.
static size_t host_region(int B, int h_q, int h_kv, int T_q, int T_kv, int d, size_t off[5]) {
  if (B < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 || T_q < 1 || T_kv < 1) return 0;
  if (d != 64 && d != 128) return 0;
  const size_t qo = static_cast<size_t>(B) * h_q * T_q * d * 2;
  const size_t kv = static_cast<size_t>(B) * h_kv * T_kv * d * 2;
  const size_t ls = static_cast<size_t>(B) * h_q * T_q * 4;
  const size_t sizes[5] = {qo, kv, kv, qo, ls};
  size_t at = 0;
  for (int i = 0; i < 5; ++i) {
    off[i] = at;
    at += (sizes[i] + 255) & ~static_cast<size_t>(255);
  }
  return at;
}

attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                            int causal, int dtype, void* device_buffer,
                            size_t device_buffer_bytes, void* stream) {
  if (h_kv < 1) return ATTN_ERR_INVALID_ARG;
  bool empty = false;
  attn_status_t st = validate(q, k, v, o, lse, B, h_q, T_q, T_kv, d, scale, causal, dtype, &empty,
                              h_kv);
  if (st != ATTN_OK) return st;
  if (empty) {
    t_last_kernel = "none";
    return ATTN_OK;
  }
  size_t off[5];
  const size_t need = host_region(B, h_q, h_kv, T_q, T_kv, d, off);
  if (need == 0) return ATTN_ERR_INVALID_ARG;
  const bool own = device_buffer == nullptr && device_buffer_bytes == 0;
  if (!own && (!device_buffer || device_buffer_bytes < need || !aligned(device_buffer, 16)))
    return ATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(device_buffer);
  if (own && cudaMallocAsync(reinterpret_cast<void**>(&base), need, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const size_t qo = static_cast<size_t>(B) * h_q * T_q * d * 2;
  const size_t kv = static_cast<size_t>(B) * h_kv * T_kv * d * 2;
  const size_t ls = static_cast<size_t>(B) * h_q * T_q * 4;
  void* dq = base + off[0];
  void* dk = base + off[1];
  void* dv = base + off[2];
  void* dO = base + off[3];
  float* dl = reinterpret_cast<float*>(base + off[4]);
  // one copy per tensor, in stream order
  if (cudaMemcpyAsync(dq, q, qo, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dk, k, kv, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dv, v, kv, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    st = ATTN_ERR_CUDA;
  } else {
    st = run(dq, dk, dv, dO, dl, B, h_q, h_kv, T_q, T_kv, d, scale, causal, dtype, 0, nullptr, 0,
             true, stream);
    if (st == ATTN_OK &&
        (cudaMemcpyAsync(o, dO, qo, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
         cudaMemcpyAsync(lse, dl, ls, cudaMemcpyDeviceToHost, s) != cudaSuccess))
      st = ATTN_ERR_CUDA;
  }
  if (own) cudaFreeAsync(base, s);
  return st;
}

attn_status_t attn_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int h, int T_q, int T_kv, int d, float scale, int causal,
                             int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  bool empty = false;
  attn_status_t st = validate(q, k, v, o, lse, B, h, T_q, T_kv, d, scale, causal, dtype, &empty);
  if (st != ATTN_OK) return st;
  if (empty) {
    t_last_kernel = "none";
    return ATTN_OK;
  }
  const long long BH = static_cast<long long>(B) * h;
  if (BH > 65535) return ATTN_ERR_UNSUPPORTED;  // one grid slice per head
  const size_t need = attn::naive_workspace_bytes(BH, T_q, T_kv);
  const bool own = workspace == nullptr && workspace_bytes == 0;
  if (!own) {
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return ATTN_ERR_WORKSPACE;
    const size_t qo = static_cast<size_t>(BH) * T_q * d * 2;
    const size_t kv = static_cast<size_t>(BH) * T_kv * d * 2;
    if (overlaps(workspace, need, q, qo) || overlaps(workspace, need, k, kv) ||
        overlaps(workspace, need, v, kv) || overlaps(workspace, need, o, qo) ||
        overlaps(workspace, need, lse, static_cast<size_t>(BH) * T_q * 4))
      return ATTN_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  if (own && cudaMallocAsync(&ws, need, s) != cudaSuccess) return ATTN_ERR_CUDA;
  attn::FwdProblem p{q, k, v, o, lse, B, h, T_q, T_kv, d, scale, causal,
                     dtype == ATTN_BF16 ? 1 : 0, nullptr, h};
  const char* name = "none";
  const cudaError_t e = attn::launch_naive(p, ws, s, &name);
  if (own) cudaFreeAsync(ws, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  t_last_kernel = name;
  return ATTN_OK;
}

size_t attn_naive_workspace_bytes(int B, int h, int T_q, int T_kv) {
  if (B < 0 || h < 0 || T_q < 0 || T_kv < 0) return 0;
  return attn::naive_workspace_bytes(static_cast<long long>(B) * h, T_q, T_kv);
}

size_t attn_host_buffer_bytes(int B, int h_q, int h_kv, int T_q, int T_kv, int d) {
  size_t off[5];
  return host_region(B, h_q, h_kv, T_q, T_kv, d, off);
}

size_t attn_splitkv_workspace_bytes(int B, int h_q, int T_q, int T_kv, int d, int num_splits) {
  if (B < 1 || h_q < 1 || T_q < 2 || T_kv < 1 || (d != 64 && d != 128)) return 0;
  if (num_splits < 0 || num_splits > 64) return 0;
  const int splits = num_splits > 0 ? num_splits : prefill_auto_splits(B, h_q, T_q, T_kv, d);
  return prefill_ws_bytes(B, h_q, T_q, d, splits);
}

size_t attn_gqa_workspace_bytes(int B, int h_q, int h_kv, int T_q, int T_kv, int d,
                                int num_splits) {
  if (B < 0 || h_q < 0 || h_kv < 1 || T_q < 0 || T_kv < 0 || (d != 64 && d != 128)) return 0;
  if (h_q % h_kv != 0) return 0;
  if (num_splits < 0 || num_splits > kMaxSplits) return 0;
  // groups of 4 or more decode on the tensor cores, which take 1..64
  // partitions (attn_fwd_gqa rejects more as unsupported)
  if (gqa_decode_on_tensor_cores(h_q, h_kv) && num_splits > 64) return 0;
  if (T_q != 1 || B == 0 || h_q == 0 || T_kv < 1) return 0;
  const int splits = num_splits > 0 ? num_splits : auto_splits(B, h_q, h_kv, T_kv, d);
  return ws_bytes(B, h_q, d, splits);
}

size_t attn_workspace_bytes(int B, int h, int T_q, int T_kv, int d, int num_splits) {
  if (B < 0 || h < 0 || T_q < 0 || T_kv < 0 || (d != 64 && d != 128)) return 0;
  if (num_splits < 0 || num_splits > kMaxSplits) return 0;
  if (T_q != 1 || B == 0 || h == 0 || T_kv < 1) return 0;
  const int splits = num_splits > 0 ? num_splits : auto_splits(B, h, h, T_kv, d);
  return ws_bytes(B, h, d, splits);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int h, int T_q, int T_kv, int d, float scale, int causal, int dtype,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, h, h, T_q, T_kv, d, scale, causal, dtype,
                 workspace, workspace_bytes, stream);
}

attn_status_t attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                           int causal, int dtype, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (h_kv < 1) return ATTN_ERR_INVALID_ARG;
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, h_q, h_kv, T_q, T_kv, d, scale, causal,
                 dtype, workspace, workspace_bytes, stream);
}

attn_status_t attn_fwd_paged_decode(const void* q, const void* k_pages, const void* v_pages,
                                    const int* block_table, const int* seq_lens, void* o,
                                    float* lse, int B, int h_q, int h_kv, int d, int page_size,
                                    int max_pages_per_seq, int num_pages, float scale, int dtype,
                                    int num_splits, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  return run_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, B, h_q, h_kv, d, page_size,
                   max_pages_per_seq, num_pages, scale, dtype, num_splits, workspace,
                   workspace_bytes, stream);
}

size_t attn_paged_workspace_bytes(int B, int h_q, int h_kv, int d, int page_size,
                                  int max_pages_per_seq, int num_splits) {
  if (B < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 || (d != 64 && d != 128) ||
      !pow2(page_size) || page_size > 65536 || max_pages_per_seq < 1 || num_splits < 0 ||
      num_splits > kMaxSplits)
    return 0;
  if (static_cast<long long>(page_size) * max_pages_per_seq > 0x7fffffffll) return 0;
  const int splits = num_splits > 0 ? num_splits
                                    : paged_auto_splits(B, h_q, h_kv, d, page_size,
                                                        max_pages_per_seq);
  if (paged_on_tensor_cores(h_q, h_kv, page_size) && splits <= 1) return 0;
  return ws_bytes(B, h_q, d, splits);
}

size_t attn_bwd_workspace_bytes(int B, int h, int T_q, int T_kv, int d) {
  if (B < 1 || h < 1 || T_q < 1 || T_kv < 1 || (d != 64 && d != 128)) return 0;
  return attn::bwd_workspace_floats(static_cast<long long>(B) * h, T_q) * sizeof(float);
}

int attn_decode_num_splits(int B, int h, int T_kv, int d) {
  if (B < 1 || h < 1 || T_kv < 1 || (d != 64 && d != 128)) return 0;
  return auto_splits(B, h, h, T_kv, d);
}

attn_status_t attn_get_device_error(void* stream, unsigned int* site) {
  if (site) *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int* p = status_ptr();
  if (!p) return ATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (site) *site = word;
  if (word == 0) return ATTN_OK;
  const unsigned int code = word & 0xffu;
  if (code == ATTN_ERR_TIMEOUT) return ATTN_ERR_TIMEOUT;
  if (code == ATTN_ERR_INVALID_ARG) return ATTN_ERR_INVALID_ARG;  // found on the device
  return ATTN_ERR_CUDA;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

attn_status_t attn_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 2000000u) return ATTN_ERR_INVALID_ARG;
  unsigned int* st = status_ptr();
  if (!st) return ATTN_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      st, static_cast<unsigned long long>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

const char* attn_last_kernel_name(void) { return t_last_kernel; }

}  // extern "C"
