// attn_internal.h -- launchers shared between the C-ABI layer (attn_api.cu)
// and the kernel translation units. Arguments arrive already validated.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "attn.h"

namespace attn {

struct FwdProblem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, h, T_q, T_kv, d;
  float scale;
  int causal;
  int bf16;               // 1 = bf16, 0 = fp16
  unsigned int* status;   // device status word of the current device
  int h_kv;               // key/value heads; h is a multiple of it (h_kv == h: plain attention)
};

// Prefill (T_q > 1): tcgen05 tensor-core kernel. With num_splits > 1 the
// key range of every query-tile pair is cut into that many partitions whose
// fp32 partials ([B*h*T_q][num_splits][d+4] at `part`) the merge kernel then
// combines into o and lse. `name` receives a static kernel name on success.
cudaError_t launch_prefill(const FwdProblem& p, int num_splits, float* part, cudaStream_t stream,
                           const char** name);

// Grouped-query decode against a paged cache on the tensor cores: the prefill
// kernel with K/V tiles gathered from the pool through the block table. p is
// the virtual problem (B, h = h_kv, T_q = G query heads per key/value head,
// T_kv = the longest length the table can name, no mask), p.k/p.v the pools.
cudaError_t launch_prefill_paged(const FwdProblem& p, const int* table, const int* lens,
                                 int page_shift, int max_pages, int num_pages, int num_splits,
                                 float* part, cudaStream_t stream, const char** name);

// The exact merge of per-row partials ([rows][S][d+4] fp32: o, m, l in log2
// units) into 16-bit o [rows][d] and lse [rows] (decode_sm103.cu).
cudaError_t launch_combine(const float* part, void* o, float* lse, long long rows, int S, int d,
                           bool bf16, cudaStream_t stream);

// Decode (T_q == 1): split kernel over `num_splits` key partitions writing
// partials to `ws`, then the merge kernel.
cudaError_t launch_decode(const FwdProblem& p, int num_splits, float* ws, cudaStream_t stream,
                          const char** name);

// Backward pass (attn_bwd): gradients dq [B,h,T_q,d], dk and dv
// [B,h_kv,T_kv,d] from q, k, v, the forward's o and lse, and dout = dO.
struct BwdProblem {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int B, h, h_kv, T_q, T_kv, d;
  float scale;
  int causal;
  int bf16;
  float* ws;              // bwd_workspace_floats(B*h, T_q) floats, 16-byte aligned
  unsigned int* status;
};

// Query rows per head in the backward workspace: T_q rounded up to 128.
inline size_t bwd_rows_padded(int T_q) { return (static_cast<size_t>(T_q) + 127) / 128 * 128; }
// Two fp32 values (lse * log2 e and rowsum(dO * O)) per padded query row.
inline size_t bwd_workspace_floats(long long BH, int T_q) {
  return 2 * static_cast<size_t>(BH) * bwd_rows_padded(T_q);
}

cudaError_t launch_backward(const BwdProblem& p, cudaStream_t stream, const char** name);

// Decode against a paged cache (attn_fwd_paged_decode): pages
// [num_pages][h_kv][page_size][d], block_table [B][max_pages] int32,
// seq_lens [B] int32 (device memory).
struct PagedProblem {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int* block_table;
  const int* seq_lens;
  void* o;
  float* lse;
  int B, h_q, h_kv, d;
  int page_shift;         // log2(page_size)
  int max_pages, num_pages;
  float scale;
  int bf16;
  unsigned int* status;
};

cudaError_t launch_decode_paged(const PagedProblem& p, int num_splits, float* ws,
                                cudaStream_t stream, const char** name);
int decode_paged_ctas_per_sm(int d);

// Query heads one CUDA-core decode split CTA serves (all sharing one
// key/value head): 2 for even groups, else 1. Groups of 4 or more query heads
// per key/value head decode on the tensor cores instead (attn_api.cu).
inline int decode_heads_per_cta(int group) { return (group % 2 == 0) ? 2 : 1; }

// The tensor-core forward pairs two heads per work unit (each with its own
// query tile and key/value stream) when a head has at most 128 query rows at
// d = 64, so that both tiles of a unit exist; its units are then
// ceil(B*h / 2) per key partition instead of B*h (contiguous or paged K/V).
inline bool head_pair_mode(int d, int T_q, long long BH) { return d == 64 && T_q <= 128 && BH >= 2; }
// With a paged cache, head pairs pay off for pages of 64 rows or more (one
// or two boxes per key tile and head); with smaller pages the producer warp's
// many box copies per key tile set the pace and one head per unit keeps more,
// smaller units (measured: 16-row pages no faster, variable lengths slower).
inline bool paged_head_pairs(int d, int T_q, long long BH, int page_size) {
  return head_pair_mode(d, T_q, BH) && page_size >= 64;
}

// Split kernel occupancy (CTAs per SM) for the split-count heuristic.
int decode_split_ctas_per_sm(int d, int heads_per_cta);

// The materialising baseline (naive_sm103.cu): S = scale * Q K^T and
// P = softmax(S), both 16-bit [B*h][T_q][T_kv], written to `workspace`
// (S first, then P), then O = P V; lse from the softmax pass.
cudaError_t launch_naive(const FwdProblem& p, void* workspace, cudaStream_t stream, const char** name);
inline size_t naive_workspace_bytes(long long BH, int T_q, int T_kv) {
  return 2 * static_cast<size_t>(BH) * static_cast<size_t>(T_q) * static_cast<size_t>(T_kv) * 2;
}

namespace detail {
// Argument checks shared by every entry point (attn_api.cu); *empty is set
// when the output has no elements.
attn_status_t validate(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                       int T_q, int T_kv, int d, float scale, int causal, int dtype, bool* empty,
                       int h_kv = -1);
// Decode split count chosen by shape on the current device (attn_api.cu):
// `rows` CTAs per partition index (B * h_kv * group / heads_per_cta).
int choose_splits(long long rows, int T_kv, int d, int heads_per_cta);
// The same rule for a given capacity (split CTAs resident on the device).
int choose_splits_cap(long long rows, int T_kv, long long cap);
}  // namespace detail

// Floats per partial: d outputs, then running max and running sum, padded
// to a 16-byte multiple.
__host__ __device__ inline constexpr size_t decode_partial_floats(int d) { return static_cast<size_t>(d) + 4; }

}  // namespace attn
