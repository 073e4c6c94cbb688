// tv_internal.h -- declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tv.h"

namespace tv {

// Cache geometry passed by value to kernels.
struct CacheGeom {
  const int32_t* page_table;  // [B, max_pages] or nullptr
  int32_t page_size;
  int32_t max_pages;
  int64_t kv_stride_b;
};

// Row of the cache holding logical key j of sequence b.
__host__ __device__ __forceinline__ int64_t cache_row(const CacheGeom& g, int b, int64_t j) {
  if (g.page_table) {
    const int32_t pg = g.page_table[(int64_t)b * g.max_pages + j / g.page_size];
    return (int64_t)pg * g.page_size + j % g.page_size;
  }
  return (int64_t)b * g.kv_stride_b + j;
}

// Store a device-detected error into the caller's status word (first writer wins is not
// guaranteed; any negative code marks the call as failed).
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicMin(status, code);
}

// Launchers (each defined next to its kernel).  Return cudaError_t of the launch.
cudaError_t launch_visibility(const int32_t* parent, int B, int Q, uint64_t* anc,
                              int32_t* depth, uint8_t* mask, int32_t* status,
                              cudaStream_t st);

cudaError_t launch_rope(const void* in, tv_dtype in_dt, int64_t isr, int64_t ish, void* out,
                        tv_dtype out_dt, int64_t osr, int64_t osh, const CacheGeom* cache,
                        int B, int Q, int NH, int D, const int32_t* prefix_len,
                        const int32_t* depth, double base, cudaStream_t st);

// Work decomposition of the SIMT attention path.
struct SimtPlan {
  int head_blocks;   // ceil(H / 32)
  int splits;        // KV splits (1 = no combine)
  int chunk;         // keys per split (multiple of 32)
};
SimtPlan simt_plan(const tv_attn_args* a, int sm_count);
size_t simt_workspace(const tv_attn_args* a, const SimtPlan& p);
bool simt_supported(const tv_attn_args* a);
cudaError_t launch_attn_simt(const tv_attn_args* a, const SimtPlan& p, void* ws,
                             cudaStream_t st);

// Work decomposition of the tensor-core path (the schedule itself is computed on the
// device from the prefix lengths).
struct TcPlan {
  int clusters;       // persistent 2-CTA clusters launched (at most)
  int tiles_per_seq;  // ceil(Q*H / 128)
  int64_t n_tiles;    // B * tiles_per_seq
  int splits;         // 0: the automatic schedule; S > 0: every tile in S pieces
  int64_t n_items;    // work items at most
  int64_t max_slots;  // partial-result slots of split tiles at most
  int64_t max_split;  // split tiles at most (records of the merge's work list)
};
bool tc_supported(const tv_attn_args* a);
TcPlan tc_plan(const tv_attn_args* a);
size_t tc_workspace(const tv_attn_args* a, const TcPlan& p);
cudaError_t launch_attn_tc(const tv_attn_args* a, const TcPlan& p, void* ws, cudaStream_t st);
int tc_launch_count(const tv_attn_args* a, const TcPlan& p);  // kernels launch_attn_tc enqueues

// Split-KV combine: partial (out_s, lse_s) for s < splits -> final out, lse.
cudaError_t launch_combine(const float* ws_out, const float* ws_lse, int splits,
                           int64_t rows, int DL, float* out, float* lse, cudaStream_t st);

// Greedy tree acceptance: argmax of every node's logits in `chunks` pieces per row, then
// the walk (k_accept.cu).
struct AcceptPlan {
  int chunks;     // pieces per logit row
  int64_t chunk;  // vocabulary entries per piece (multiple of 2048)
};
AcceptPlan accept_plan(int B, int Q, int64_t V, int sm_count);
size_t accept_workspace(int B, int Q, const AcceptPlan& p);
cudaError_t launch_accept(const void* logits, tv_dtype dt, int64_t V, int64_t stride,
                          const int32_t* parent, const int32_t* tokens, int B, int Q,
                          int32_t* target, int32_t* accept_len, int32_t* path,
                          int32_t* new_tokens, int32_t* status, const AcceptPlan& p,
                          void* ws, cudaStream_t st);
// Post-verify compaction of the accepted nodes' cache rows (k_accept.cu); strides and row
// sizes in bytes, multiples of 16.
cudaError_t launch_compact(void* c_kv, int64_t ckv_stride_bytes, void* k_pe,
                           int64_t kpe_stride_bytes, int ckv_row_bytes, int kpe_row_bytes,
                           const CacheGeom& g, int64_t num_rows, const int32_t* prefix_len,
                           const int32_t* path, const int32_t* accept_len, int B, int Q,
                           int32_t* new_prefix_len, int32_t* status, cudaStream_t st);

// The fused steps before the attention (k_prologue.cu).
cudaError_t launch_prologue(const tv_prologue_args* a, cudaStream_t st);

// Best-first draft-tree construction (k_tree.cu).
cudaError_t launch_build_tree(const float* lp, const int32_t* tok, const int32_t* root, int B,
                              int L, int K, int budget, int32_t* parent, int32_t* tokens,
                              int32_t* depth, float* score, int32_t* status, cudaStream_t st);

// Set the thread-local text returned by tv_last_error() (defined in tv_api.cu).
void set_last_error(const char* msg);

// Number of SMs of the current device (148 if it cannot be queried).
int current_sm_count();

}  // namespace tv
