// tv_api.cu -- the C ABI of libtv (include/tv.h): argument checks, path choice, launches.
//
// Every entry point validates its arguments on the host, then enqueues its kernels on
// the caller's stream.  Nothing here allocates device memory or synchronises.
#include <cuda_runtime.h>

#include <cstdio>
#include <string>

#include "tv.h"
#include "tv_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, const char* detail = "") {
  char buf[512];
  snprintf(buf, sizeof(buf), fmt, detail);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  char buf[512];
  snprintf(buf, sizeof(buf), "%s: %s", where, cudaGetErrorString(e));
  g_last_error = buf;
  return TV_ERR_CUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

int check_attn(const tv_attn_args* a) {
  if (!a) return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: args is NULL%s");
  if (a->struct_size != sizeof(tv_attn_args))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: struct_size mismatch (ABI)%s");
  if (a->B < 0 || a->H < 1 || a->Q < 1 || a->d_latent < 8 || a->d_rope < 0)
    return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: bad B/H/Q/d_latent/d_rope%s");
  if (a->mask_mode != TV_MASK_TREE && a->mask_mode != TV_MASK_CAUSAL)
    return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: bad mask_mode%s");
  const bool causal = a->mask_mode == TV_MASK_CAUSAL;
  if (a->Q > 64 && !causal)
    return fail(TV_ERR_UNSUPPORTED, "tv_verify_attn: Q > 64 needs TV_MASK_CAUSAL%s");
  if ((int64_t)a->B * a->Q * a->H >= (1ll << 31))
    return fail(TV_ERR_UNSUPPORTED, "tv_verify_attn: B*Q*H must be below 2^31%s");
  if (a->d_latent % 8 || a->d_rope % 8)
    return fail(TV_ERR_UNSUPPORTED, "tv_verify_attn: d_latent and d_rope must be multiples of 8%s");
  if (!(a->q_dt == TV_F32 || a->q_dt == TV_BF16) || a->q_dt != a->kv_dt)
    return fail(TV_ERR_UNSUPPORTED, "tv_verify_attn: q_dt and kv_dt must both be F32 or BF16%s");
  if (a->max_prefix_len < 0) return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: max_prefix_len < 0%s");
  if (a->B == 0) return TV_OK;
  if (!a->q_latent || !a->c_kv || !a->prefix_len || (!causal && !a->anc) || !a->out || !a->lse ||
      (a->d_rope > 0 && (!a->q_pe || !a->k_pe)))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: NULL tensor pointer%s");
  const int64_t es = a->kv_dt == TV_BF16 ? 2 : 4;
  if (a->ckv_row_stride < a->d_latent || (a->d_rope > 0 && a->kpe_row_stride < a->d_rope))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: row stride smaller than the row%s");
  if (!aligned16(a->c_kv) || (a->ckv_row_stride * es) % 16 ||
      (a->d_rope > 0 && (!aligned16(a->k_pe) || (a->kpe_row_stride * es) % 16)) ||
      !aligned16(a->q_latent) || (a->d_rope > 0 && !aligned16(a->q_pe)) || !aligned16(a->out))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: tensors and rows must be 16-byte aligned%s");
  const int64_t kv_max = (int64_t)a->max_prefix_len + a->Q;
  if (a->cache.page_table) {
    if (a->cache.page_size <= 0 || a->cache.max_pages <= 0)
      return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: paged cache needs page_size and max_pages%s");
    if (kv_max > (int64_t)a->cache.page_size * a->cache.max_pages)
      return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: max_prefix_len + Q exceeds max_pages*page_size%s");
  } else if (a->cache.kv_stride_b < kv_max) {
    return fail(TV_ERR_INVALID_ARG, "tv_verify_attn: kv_stride_b < max_prefix_len + Q%s");
  }
  if (a->path < TV_PATH_AUTO || a->path > TV_PATH_TCGEN05 || a->num_splits < 0 ||
      a->paged_view < TV_PAGED_AUTO || a->paged_view > TV_PAGED_GATHER ||
      (a->overlap_prev != 0 && a->overlap_prev != 1))
    return fail(TV_ERR_INVALID_ARG,
                "tv_verify_attn: bad path, num_splits, paged_view or overlap_prev%s");
  return TV_OK;
}

// Tensor cores when the shape is the absorbed-MLA one they implement (bf16, d_latent 512,
// d_rope 64, known cache size) and the problem has at least two full 128-row tiles;
// CUDA cores otherwise.
int resolve_path(const tv_attn_args* a) {
  const bool tc_ok = tv::tc_supported(a);
  if (a->path == TV_PATH_TCGEN05) {
    if (!tc_ok)
      return fail(TV_ERR_UNSUPPORTED,
                  "tv_verify_attn: tensor-core path needs bf16 q and cache, d_latent 512, "
                  "d_rope 64, 64-token pages and cache.num_rows%s");
    return TV_PATH_TCGEN05;
  }
  if (a->path == TV_PATH_AUTO && tc_ok && (int64_t)a->B * a->Q * a->H >= 256)
    return TV_PATH_TCGEN05;
  if (!tv::simt_supported(a))
    return fail(TV_ERR_UNSUPPORTED, "tv_verify_attn: shape not supported%s");
  return TV_PATH_SIMT;
}

}  // namespace

namespace tv {
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }
int current_sm_count() { return sm_count(); }
}  // namespace tv

extern "C" {

int tv_version(void) { return 100; }

const char* tv_status_string(int code) {
  switch (code) {
    case TV_OK: return "ok";
    case TV_ERR_INVALID_ARG: return "invalid argument";
    case TV_ERR_INVALID_TREE: return "invalid draft-tree parent array";
    case TV_ERR_UNSUPPORTED: return "unsupported request";
    case TV_ERR_CUDA: return "CUDA error";
    case TV_ERR_TIMEOUT: return "device wait timed out";
    case TV_ERR_WORKSPACE: return "workspace missing or too small";
    case TV_ERR_BOUNDS: return "prefix length outside the cache geometry";
    default: return "unknown status";
  }
}

const char* tv_last_error(void) { return g_last_error.c_str(); }

int tv_build_visibility(const int32_t* parent, int B, int Q, uint64_t* anc, int32_t* depth,
                        uint8_t* dense_mask, int32_t* status, void* stream) {
  g_last_error.clear();
  if (B < 0 || Q < 1) return fail(TV_ERR_INVALID_ARG, "tv_build_visibility: B < 0 or Q < 1%s");
  if (Q > 64) return fail(TV_ERR_UNSUPPORTED, "tv_build_visibility: Q > 64 not supported%s");
  if (B > 0 && (!parent || !anc || !depth))
    return fail(TV_ERR_INVALID_ARG, "tv_build_visibility: NULL pointer%s");
  cudaError_t e = tv::launch_visibility(parent, B, Q, anc, depth, dense_mask, status,
                                        (cudaStream_t)stream);
  return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_build_visibility");
}

int tv_rope_neox(const void* in, tv_dtype in_dt, int64_t in_stride_row,
                 int64_t in_stride_head, void* out, tv_dtype out_dt, int64_t out_stride_row,
                 int64_t out_stride_head, const tv_cache_layout* out_cache, int B, int Q,
                 int n_heads, int d_rope, const int32_t* prefix_len, const int32_t* depth,
                 double base, void* stream) {
  g_last_error.clear();
  if (B < 0 || Q < 1 || n_heads < 1 || d_rope <= 0 || (d_rope & 1) || d_rope > 512)
    return fail(TV_ERR_INVALID_ARG, "tv_rope_neox: bad B/Q/n_heads/d_rope%s");
  if (!(in_dt == TV_F32 || in_dt == TV_BF16) || !(out_dt == TV_F32 || out_dt == TV_BF16))
    return fail(TV_ERR_INVALID_ARG, "tv_rope_neox: bad dtype%s");
  if (!(base > 0.0)) return fail(TV_ERR_INVALID_ARG, "tv_rope_neox: base must be > 0%s");
  if (B == 0) return TV_OK;
  if (!in || !out || !prefix_len)
    return fail(TV_ERR_INVALID_ARG, "tv_rope_neox: NULL pointer%s");
  if (in_stride_head < d_rope || out_stride_head < d_rope ||
      in_stride_row < (int64_t)(n_heads - 1) * in_stride_head + d_rope ||
      out_stride_row < (int64_t)(n_heads - 1) * out_stride_head + d_rope)
    return fail(TV_ERR_INVALID_ARG, "tv_rope_neox: strides make rows or heads overlap%s");
  tv::CacheGeom g{};
  if (out_cache) {
    g = tv::CacheGeom{out_cache->page_table, out_cache->page_size, out_cache->max_pages,
                      out_cache->kv_stride_b};
    if (g.page_table && (g.page_size <= 0 || g.max_pages <= 0))
      return fail(TV_ERR_INVALID_ARG, "tv_rope_neox: paged cache needs page_size and max_pages%s");
    if (!g.page_table && g.kv_stride_b < Q)
      return fail(TV_ERR_INVALID_ARG, "tv_rope_neox: kv_stride_b too small%s");
  }
  cudaError_t e = tv::launch_rope(in, in_dt, in_stride_row, in_stride_head, out, out_dt,
                                  out_stride_row, out_stride_head, out_cache ? &g : nullptr,
                                  B, Q, n_heads, d_rope, prefix_len, depth, base,
                                  (cudaStream_t)stream);
  return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_rope_neox");
}

int tv_verify_attn_path(const tv_attn_args* a) {
  g_last_error.clear();
  int rc = check_attn(a);
  if (rc != TV_OK) return rc;
  return resolve_path(a);
}

int tv_verify_attn_launches(const tv_attn_args* a) {
  const int path = tv_verify_attn_path(a);
  if (path < 0) return path;
  if (path == TV_PATH_TCGEN05) return tv::tc_launch_count(a, tv::tc_plan(a));
  return 1 + (tv::simt_plan(a, sm_count()).splits > 1 ? 1 : 0);
}

size_t tv_verify_attn_workspace_size(const tv_attn_args* a) {
  if (check_attn(a) != TV_OK) return 0;
  const int path = resolve_path(a);
  if (path == TV_PATH_SIMT) return tv::simt_workspace(a, tv::simt_plan(a, sm_count()));
  if (path == TV_PATH_TCGEN05) return tv::tc_workspace(a, tv::tc_plan(a));
  return 0;
}

int tv_verify_attn(const tv_attn_args* a, void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  int rc = check_attn(a);
  if (rc != TV_OK) return rc;
  if (a->B == 0) return TV_OK;
  const int path = resolve_path(a);
  if (path < 0) return path;
  if (workspace && ((uintptr_t)workspace & 255u))
    return fail(TV_ERR_WORKSPACE, "tv_verify_attn: workspace must be 256-byte aligned%s");
  if (path == TV_PATH_TCGEN05) {
    const tv::TcPlan plan = tv::tc_plan(a);
    const size_t need = tv::tc_workspace(a, plan);
    if (need > 0 && (!workspace || ws_bytes < need))
      return fail(TV_ERR_WORKSPACE, "tv_verify_attn: workspace smaller than tv_verify_attn_workspace_size()%s");
    cudaError_t e = tv::launch_attn_tc(a, plan, workspace, (cudaStream_t)stream);
    return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_verify_attn (tensor cores)");
  }
  const tv::SimtPlan plan = tv::simt_plan(a, sm_count());
  const size_t need = tv::simt_workspace(a, plan);
  if (need > 0 && (!workspace || ws_bytes < need))
    return fail(TV_ERR_WORKSPACE, "tv_verify_attn: workspace smaller than tv_verify_attn_workspace_size()%s");
  cudaError_t e = tv::launch_attn_simt(a, plan, workspace, (cudaStream_t)stream);
  return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_verify_attn");
}

int tv_verify_prologue(const tv_prologue_args* a, void* stream) {
  g_last_error.clear();
  if (!a) return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: args is NULL%s");
  if (a->struct_size != sizeof(tv_prologue_args))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: struct_size mismatch (ABI)%s");
  if (a->B < 0 || a->Q < 1 || a->H < 1 || a->d_rope <= 0 || a->d_latent < 0)
    return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: bad B/Q/H/d_rope/d_latent%s");
  if (a->Q > 64) return fail(TV_ERR_UNSUPPORTED, "tv_verify_prologue: Q > 64 not supported%s");
  if (a->d_rope % 8 || a->d_rope > 512 || a->d_latent % 8)
    return fail(TV_ERR_UNSUPPORTED, "tv_verify_prologue: d_rope and d_latent must be multiples of 8, d_rope <= 512%s");
  if ((int64_t)a->H * a->d_rope > 8192)
    return fail(TV_ERR_UNSUPPORTED, "tv_verify_prologue: H * d_rope must be at most 8192%s");
  if (!(a->q_dt == TV_F32 || a->q_dt == TV_BF16) || !(a->kv_dt == TV_F32 || a->kv_dt == TV_BF16))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: bad dtype%s");
  if (!(a->rope_base > 0.0)) return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: rope_base must be > 0%s");
  if (a->B == 0) return TV_OK;
  if (!a->parent || !a->prefix_len || !a->q_pe_in || !a->q_pe_out || !a->kpe_tree || !a->k_pe ||
      !a->anc || !a->depth || (a->ckv_tree && !a->c_kv))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: NULL pointer%s");
  const int64_t ek = a->kv_dt == TV_BF16 ? 2 : 4;
  if (!aligned16(a->q_pe_in) || !aligned16(a->q_pe_out) || !aligned16(a->kpe_tree) ||
      !aligned16(a->k_pe) || (a->kpe_row_stride * ek) % 16 || a->kpe_row_stride < a->d_rope ||
      (a->ckv_tree && (!aligned16(a->ckv_tree) || !aligned16(a->c_kv) ||
                       (a->ckv_row_stride * ek) % 16 || a->ckv_row_stride < a->d_latent)))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: tensors and rows must be 16-byte aligned%s");
  if (a->cache.page_table && (a->cache.page_size <= 0 || a->cache.max_pages <= 0))
    return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: paged cache needs page_size and max_pages%s");
  if (!a->cache.page_table && a->cache.kv_stride_b < a->Q)
    return fail(TV_ERR_INVALID_ARG, "tv_verify_prologue: kv_stride_b too small%s");
  cudaError_t e = tv::launch_prologue(a, (cudaStream_t)stream);
  return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_verify_prologue");
}

int tv_build_tree(const float* logprobs, const int32_t* cand_tokens, const int32_t* root_token,
                  int B, int L, int K, int budget, int32_t* parent, int32_t* tokens,
                  int32_t* depth, float* score, int32_t* status, void* stream) {
  g_last_error.clear();
  if (B < 0 || L < 1 || K < 1 || budget < 0)
    return fail(TV_ERR_INVALID_ARG, "tv_build_tree: bad B/L/K/budget%s");
  if (L > 16 || K > 16 || budget > 63)
    return fail(TV_ERR_UNSUPPORTED, "tv_build_tree: needs L <= 16, K <= 16, budget <= 63%s");
  double paths = 0.0, level = 1.0;
  for (int d = 1; d <= L; ++d) {
    level *= K;
    paths += level;
  }
  if ((double)budget > paths)
    return fail(TV_ERR_INVALID_ARG, "tv_build_tree: budget exceeds the possible nodes%s");
  if (B == 0) return TV_OK;
  if (!logprobs || !cand_tokens || !parent || !tokens)
    return fail(TV_ERR_INVALID_ARG, "tv_build_tree: NULL pointer%s");
  cudaError_t e = tv::launch_build_tree(logprobs, cand_tokens, root_token, B, L, K, budget,
                                        parent, tokens, depth, score, status,
                                        (cudaStream_t)stream);
  return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_build_tree");
}

size_t tv_tree_accept_workspace_size(int B, int Q, int64_t vocab) {
  if (B < 0 || Q < 1 || Q > 64 || vocab < 1) return 0;
  return tv::accept_workspace(B, Q, tv::accept_plan(B, Q, vocab, sm_count()));
}

int tv_tree_accept(const void* logits, tv_dtype logits_dt, int64_t vocab,
                   int64_t logits_row_stride, const int32_t* parent, const int32_t* tokens,
                   int B, int Q, int32_t* target, int32_t* accept_len, int32_t* path,
                   int32_t* new_tokens, int32_t* status, void* workspace, size_t ws_bytes,
                   void* stream) {
  g_last_error.clear();
  if (B < 0 || Q < 1) return fail(TV_ERR_INVALID_ARG, "tv_tree_accept: B < 0 or Q < 1%s");
  if (Q > 64) return fail(TV_ERR_UNSUPPORTED, "tv_tree_accept: Q > 64 not supported%s");
  if (!(logits_dt == TV_F32 || logits_dt == TV_BF16))
    return fail(TV_ERR_INVALID_ARG, "tv_tree_accept: logits must be F32 or BF16%s");
  if (vocab < 1 || vocab >= 0x7FFFFFFFll || logits_row_stride < vocab)
    return fail(TV_ERR_INVALID_ARG, "tv_tree_accept: bad vocab or row stride%s");
  if (B == 0) return TV_OK;
  if (!logits || !parent || !tokens || !accept_len || !path || !new_tokens)
    return fail(TV_ERR_INVALID_ARG, "tv_tree_accept: NULL pointer%s");
  const uintptr_t es = logits_dt == TV_BF16 ? 2 : 4;
  if ((uintptr_t)logits % es)
    return fail(TV_ERR_INVALID_ARG, "tv_tree_accept: logits not aligned to its element size%s");
  const tv::AcceptPlan plan = tv::accept_plan(B, Q, vocab, sm_count());
  const size_t need = tv::accept_workspace(B, Q, plan);
  if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < need)
    return fail(TV_ERR_WORKSPACE, "tv_tree_accept: workspace missing, misaligned or smaller "
                                  "than tv_tree_accept_workspace_size()%s");
  cudaError_t e = tv::launch_accept(logits, logits_dt, vocab, logits_row_stride, parent, tokens,
                                    B, Q, target, accept_len, path, new_tokens, status, plan,
                                    workspace, (cudaStream_t)stream);
  return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_tree_accept");
}

int tv_compact_kv(void* c_kv, void* k_pe, tv_dtype kv_dt, int64_t ckv_row_stride,
                  int64_t kpe_row_stride, int d_latent, int d_rope,
                  const tv_cache_layout* cache, const int32_t* prefix_len, const int32_t* path,
                  const int32_t* accept_len, int B, int Q, int32_t* new_prefix_len,
                  int32_t* status, void* stream) {
  g_last_error.clear();
  if (B < 0 || Q < 1 || d_latent < 0 || d_rope < 0)
    return fail(TV_ERR_INVALID_ARG, "tv_compact_kv: bad B/Q/d_latent/d_rope%s");
  if (Q > 64) return fail(TV_ERR_UNSUPPORTED, "tv_compact_kv: Q > 64 not supported%s");
  if (!(kv_dt == TV_F32 || kv_dt == TV_BF16))
    return fail(TV_ERR_INVALID_ARG, "tv_compact_kv: bad dtype%s");
  if (!cache || cache->num_rows <= 0)
    return fail(TV_ERR_INVALID_ARG, "tv_compact_kv: cache layout with num_rows is required%s");
  if (B == 0) return TV_OK;
  if (!c_kv || (d_rope > 0 && !k_pe) || !prefix_len || !path || !accept_len || !new_prefix_len)
    return fail(TV_ERR_INVALID_ARG, "tv_compact_kv: NULL pointer%s");
  const int64_t es = kv_dt == TV_BF16 ? 2 : 4;
  if (ckv_row_stride < d_latent || (d_rope > 0 && kpe_row_stride < d_rope) ||
      (d_latent * es) % 16 || (d_rope * es) % 16 || (ckv_row_stride * es) % 16 ||
      (d_rope > 0 && (kpe_row_stride * es) % 16) || !aligned16(c_kv) ||
      (d_rope > 0 && !aligned16(k_pe)))
    return fail(TV_ERR_INVALID_ARG,
                "tv_compact_kv: rows, strides and pointers must be 16-byte multiples%s");
  tv::CacheGeom g{cache->page_table, cache->page_size, cache->max_pages, cache->kv_stride_b};
  if (g.page_table && (g.page_size <= 0 || g.max_pages <= 0))
    return fail(TV_ERR_INVALID_ARG, "tv_compact_kv: paged cache needs page_size and max_pages%s");
  if (!g.page_table && g.kv_stride_b < Q)
    return fail(TV_ERR_INVALID_ARG, "tv_compact_kv: kv_stride_b too small%s");
  cudaError_t e = tv::launch_compact(c_kv, ckv_row_stride * es, d_rope > 0 ? k_pe : c_kv,
                                     kpe_row_stride * es, (int)(d_latent * es),
                                     (int)(d_rope * es), g, cache->num_rows, prefix_len, path,
                                     accept_len, B, Q, new_prefix_len, status,
                                     (cudaStream_t)stream);
  return e == cudaSuccess ? TV_OK : cuda_fail(e, "tv_compact_kv");
}

}  // extern "C"
