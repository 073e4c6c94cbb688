/*
 * tv.h -- C ABI of libtv: GB300 (sm_103a) tree-verify MLA-absorb attention for DDTree
 * speculative decoding.
 *
 * The operations come from three web pages about a native DDTree engine:
 *   [RoPE]   "Precision as Correctness: The Float64 RoPE Decision in a Custom CUDA
 *             Inference Engine"
 *   [VERIFY] "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA
 *             Attention Kernel"
 *   [GOLDEN] "The Golden Reference: A Pivotal Moment in Building a Native DDTree
 *             Inference Engine"
 *
 * One verify step of a draft tree with q_len = Q nodes (node 0 is the root) over a
 * sequence whose cache already holds prefix_len = P tokens is:
 *   1. tv_build_visibility: parent array -> ancestor-or-self bitsets and depths;
 *   2. tv_rope_neox: NeoX RoPE at position P + depth on the queries' rope part, and on the
 *      draft tokens' k_pe rows, which it writes into cache slots P + node;
 *   3. tv_verify_attn: for every (sequence, node, head), softmax attention in latent
 *      space over the P prefix keys plus the node's ancestor-or-self tree keys, returning
 *      the softmax-weighted sum of latent rows and the log-sum-exp of the scores.
 *
 * Conventions (every entry point):
 *   - Tensor pointers are DEVICE pointers owned by the caller, unless stated otherwise.
 *     The library allocates no device memory; scratch is a caller-provided workspace.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     The return value reports synchronous argument checks and launch errors only.
 *   - Calls make no synchronising CUDA call, so they can be captured into a CUDA graph on
 *     a capturing stream.  The first call in a process (or on a new device) does one-time
 *     set-up (occupancy query, driver entry points); make it outside a capture.  A graph
 *     keeps the call's arguments, sizes and workspace as they were when it was captured.
 *   - Data-dependent errors found on the device (an invalid parent array, a prefix that
 *     does not fit the cache geometry, a device wait that ran out) are stored as a
 *     negative tv_status into *status, a caller-owned device int32.  The library never
 *     clears it: set it to TV_OK before the first call and read it when convenient.
 *     `status` may be NULL, in which case such errors are dropped silently.
 *   - On a non-OK return, tv_last_error() (thread-local) describes the failure.
 *   - Element strides are in ELEMENTS, not bytes.
 */
#ifndef TV_H_
#define TV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TV_OK = 0,
  TV_ERR_INVALID_ARG = -1,  /* a pointer, size or stride is invalid */
  TV_ERR_INVALID_TREE = -2, /* parent[0] != -1 or parent[i] outside [0, i) */
  TV_ERR_UNSUPPORTED = -3,  /* valid but outside what the library implements (Q > 64 ...) */
  TV_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed (see tv_last_error) */
  TV_ERR_TIMEOUT = -5,      /* a bounded device-side wait gave up (device status only) */
  TV_ERR_WORKSPACE = -6,    /* workspace missing or smaller than the size query asked for */
  TV_ERR_BOUNDS = -7        /* prefix_len[b] + Q exceeds the cache geometry (device) */
} tv_status;

typedef enum { TV_F32 = 0, TV_BF16 = 1 } tv_dtype;

/* Kernel family for tv_verify_attn.  AUTO picks by shape and dtype; the others force one
 * family (used by tests to check both) and fail with TV_ERR_UNSUPPORTED when it cannot
 * run the request. */
typedef enum { TV_PATH_AUTO = 0, TV_PATH_SIMT = 1, TV_PATH_TCGEN05 = 2 } tv_path;

/* How the tensor-core path reads a paged cache.  AUTO (and TV_PAGED_STEP_MAPS) builds two
 * tensor maps per 128-key step that read the two 64-token pages of the step in place;
 * TV_PAGED_GATHER first copies the pages into a contiguous key view in the workspace
 * (needs B * (max_prefix_len + Q rounded up to 128) < 2^31 rows, else the maps are used).
 * Ignored by the CUDA-core path and by contiguous caches. */
typedef enum { TV_PAGED_AUTO = 0, TV_PAGED_STEP_MAPS = 1, TV_PAGED_GATHER = 2 } tv_paged_view;

/* Which keys a query row sees (tv_attn_args.mask_mode).  [GOLDEN] §"Principled
 * Abstraction": one forward_tokens call serves tree verification, autoregressive decoding
 * (one query, every key) and prefill (causal masking).
 *   TV_MASK_TREE   : node i sees the P prefix keys and its ancestor-or-self tree keys
 *                    (anc bitsets from tv_build_visibility; Q <= 64);
 *   TV_MASK_CAUSAL : query token i (at logical key P + i) sees keys 0 .. P + i: prefill of
 *                    Q tokens after a cache of P (P = 0: no prior cache); anc is not read
 *                    and may be NULL; Q is limited only by B*Q*H < 2^31. */
typedef enum { TV_MASK_TREE = 0, TV_MASK_CAUSAL = 1 } tv_mask_mode;

/*
 * Geometry of the latent KV cache.  Logical key j (0 <= j < prefix_len[b] + Q) of
 * sequence b lives in cache row
 *     page_table[b*max_pages + j/page_size]*page_size + j%page_size   (paged), or
 *     b*kv_stride_b + j                                                (page_table NULL).
 * The draft-tree token of node i occupies logical key prefix_len[b] + i.  ([GOLDEN]
 * §"Recursive Refinement of the Decode Loop Design" works out the cache slots of the root
 * and draft tokens without printing a formula; the reading taken here is that the tree
 * tokens follow the prefix in node order.)  Paged caches need page_size == 64 on the
 * tensor-core path.
 */
typedef struct {
  const int32_t* page_table; /* device [B, max_pages] int32, or NULL for contiguous */
  int32_t page_size;         /* tokens per page (paged layout) */
  int32_t max_pages;         /* row stride of page_table, pages per sequence at most */
  int64_t kv_stride_b;       /* contiguous layout: cache rows per sequence */
  int64_t num_rows;          /* rows in the c_kv / k_pe arrays; bounds the tensor-core
                                path's TMA reads (0 = unknown: that path is not used) */
} tv_cache_layout;

/*
 * tv_build_visibility -- ancestor-or-self bitsets of a draft tree.
 *
 * [VERIFY] §Context: the verify kernel applies a visibility mask that decides which tree
 * tokens each query may attend to; [GOLDEN] §"Principled Abstraction": the step is M query
 * tokens against the cache under an [M, kv_len] mask.  Each node sees its ancestors and
 * itself.
 *
 * parent     : device [B, Q] int32, topologically ordered: parent[b*Q] == -1 and
 *              0 <= parent[b*Q+i] < i for i > 0.
 * anc        : device [B, Q] uint64 out; bit k of anc[b*Q+i] is set iff node k is node i or
 *              one of its ancestors.
 * depth      : device [B, Q] int32 out; parent steps from node i to the root.
 * dense_mask : device [B, Q, Q] uint8 out, nullable; dense_mask[(b*Q+i)*Q+k] = bit k of
 *              anc[b*Q+i].
 * status     : see the conventions above.  A sequence with an invalid parent array gets
 *              anc = 0, depth = -1 (and an all-zero mask row) and TV_ERR_INVALID_TREE.
 * Returns TV_ERR_UNSUPPORTED for Q > 64 (one 64-bit word per node), TV_ERR_INVALID_ARG
 * for B < 0, Q < 1 or a NULL parent/anc/depth with B > 0.
 */
int tv_build_visibility(const int32_t* parent, int B, int Q, uint64_t* anc, int32_t* depth,
                        uint8_t* dense_mask, int32_t* status, void* stream);

/*
 * tv_rope_neox -- NeoX (rotate-half) rotary embedding with a float64 angle.
 *
 * [RoPE] §"The Message" and §"What Input Knowledge Is Required" (item 1): split the rope
 * vector in half and rotate each pair (k, k + d_rope/2) by cos/sin of the angle;
 * §"The Float64 Decision": the angle and the trigonometry run in double precision and the
 * result is converted to float32 at the end.  Here the rotation itself is also done in
 * double, so the float32 result carries one rounding; bf16 output rounds that float32
 * value to nearest-even once more.
 *
 * For every (b, i, h), with pos = prefix_len[b] + depth[b*Q+i] and, for k < d_rope/2,
 * inv_k = 1 / base^(2k/d_rope), a = pos * inv_k:
 *     out[k]          = in[k] cos a - in[k + d/2] sin a
 *     out[k + d/2]    = in[k + d/2] cos a + in[k] sin a
 *
 * in  : element (b, i, h, r) at in[(b*Q+i)*in_stride_row + h*in_stride_head + r].
 * out : element (b, i, h, r) at out[row*out_stride_row + h*out_stride_head + r] where
 *       row = b*Q+i when out_cache is NULL, else the cache row of logical key
 *       prefix_len[b] + i under *out_cache (host struct; the draft tokens' k_pe rows are
 *       rotated straight into their cache slots).  in == out with equal strides is
 *       allowed (in place).
 * in_dt / out_dt : TV_F32 or TV_BF16 each.
 * prefix_len [B], depth [B, Q]: device int32 (depth from tv_build_visibility; a negative
 *       depth -- an invalid tree -- leaves that row untouched).  depth may be NULL: then
 *       row i is at position prefix_len[b] + i (a chain of tokens, as in prefill).  With out_cache, rows whose
 *       slot lies outside the geometry (negative prefix_len, a page index >= max_pages, a
 *       negative page-table entry, or a slot >= kv_stride_b) are skipped.
 * Returns TV_ERR_INVALID_ARG for odd or non-positive d_rope, n_heads < 1, or strides
 * that make rows overlap.
 */
int tv_rope_neox(const void* in, tv_dtype in_dt, int64_t in_stride_row,
                 int64_t in_stride_head, void* out, tv_dtype out_dt, int64_t out_stride_row,
                 int64_t out_stride_head, const tv_cache_layout* out_cache, int B, int Q,
                 int n_heads, int d_rope, const int32_t* prefix_len, const int32_t* depth,
                 double base, void* stream);

/*
 * Arguments of tv_verify_attn (absorbed-MLA tree-verify attention).
 *
 * [VERIFY] §"Input Knowledge Required" and [GOLDEN] §"The Absorb Form of MLA": the key
 * projection is folded into the query, so the score of query row (b, i, h) against key j
 * is taken in latent space:
 *     s_j = scale * ( q_latent[b,i,h,:] . c_kv[j,:]  +  q_pe[b,i,h,:] . k_pe[j,:] )
 * over the visible keys V = { j < P_b } U { P_b + k : bit k of anc[b*Q+i] }, and
 *     out[b,i,h,:] = sum_{j in V} softmax(s)_j * c_kv[j,:],   lse[b,i,h] = ln sum exp(s_j).
 * With mask_mode = TV_MASK_CAUSAL the visible set is V = { j <= P_b + i } instead (prefill;
 * Q > 64 allowed, anc unused).
 */
typedef struct {
  uint32_t struct_size;     /* sizeof(tv_attn_args): ABI check */
  int32_t B, H, Q;          /* batch, heads, q_len (tree nodes, 1..64) */
  int32_t d_latent, d_rope; /* d_latent % 8 == 0, d_rope % 8 == 0 (vector loads) */
  float scale;              /* softmax scale */
  tv_dtype q_dt, kv_dt;     /* (F32, F32) or (BF16, BF16) */
  const void* q_latent;     /* [B, Q, H, d_latent] contiguous */
  const void* q_pe;         /* [B, Q, H, d_rope] contiguous, RoPE already applied */
  const void* c_kv;         /* cache rows, row r at c_kv + r*ckv_row_stride (16 B aligned) */
  const void* k_pe;         /* cache rows, row r at k_pe + r*kpe_row_stride (16 B aligned) */
  int64_t ckv_row_stride, kpe_row_stride; /* elements; rows 16-byte aligned */
  tv_cache_layout cache;    /* where key j of sequence b lives */
  const int32_t* prefix_len; /* device [B] int32, 0 <= prefix_len[b] <= max_prefix_len */
  int32_t max_prefix_len;   /* host-side bound on prefix_len, sizes the launch */
  const uint64_t* anc;      /* device [B, Q] from tv_build_visibility */
  float* out;               /* device [B, Q, H, d_latent] float32 out */
  float* lse;               /* device [B, Q, H] float32 out (natural log) */
  int32_t* status;          /* device int32, nullable (see conventions) */
  int32_t path;             /* tv_path; TV_PATH_AUTO normally */
  int32_t num_splits;       /* 0 = automatic; else cut every KV sweep into this many
                               pieces (tensor cores: each 128-row tile's sweep) */
  int32_t paged_view;       /* tv_paged_view; TV_PAGED_AUTO normally */
  int32_t mask_mode;        /* tv_mask_mode; TV_MASK_TREE for tree verification */
  int32_t overlap_prev;     /* 0 normally.  1: the work queued on the stream before this call
                               writes none of prefix_len and the page table (as for
                               tv_verify_prologue, which writes q_pe, cache rows and anc);
                               the tensor-core path's preparation kernel (work schedule,
                               per-step tensor maps) may then run while that work finishes.
                               The attention itself still starts only after all of it. */
} tv_attn_args;

/* Bytes of workspace tv_verify_attn needs for these arguments (0 if none).  The size
 * depends on B, H, Q, d_latent, max_prefix_len, whether the cache is paged, the path,
 * num_splits and paged_view only (the tensor-core path of a paged cache keeps two tensor
 * maps per 128-key step there, or with TV_PAGED_GATHER a contiguous copy of the keys). */
size_t tv_verify_attn_workspace_size(const tv_attn_args* a);

/* The kernel family TV_PATH_AUTO resolves to for these arguments, or a negative
 * tv_status if the arguments are invalid. */
int tv_verify_attn_path(const tv_attn_args* a);

/* How many kernels one tv_verify_attn call with these arguments enqueues (for launch
 * accounting; the CUDA-core path: attention + split combine; the tensor-core path: work
 * preparation + key gather (TV_PAGED_GATHER only) + attention + the merge of split tiles
 * unless num_splits == 1), or a negative tv_status if the arguments are invalid. */
int tv_verify_attn_launches(const tv_attn_args* a);

/*
 * tv_verify_attn -- run the attention.  workspace: device memory of at least
 * tv_verify_attn_workspace_size(a) bytes, 256-byte aligned (NULL allowed when the size
 * is 0); it is scratch and may be reused once the call's work on `stream` is done.
 * Rows of a sequence whose prefix_len is negative or does not fit the cache geometry get
 * out = 0, lse = -inf and TV_ERR_BOUNDS in *status.  Page-table entries of the pages that
 * hold keys 0 .. prefix_len[b]+Q-1 must name valid cache pages (they are not checked).
 */
int tv_verify_attn(const tv_attn_args* a, void* workspace, size_t ws_bytes, void* stream);

/*
 * tv_verify_attn_noalloc -- tv_verify_attn for callers that cannot allocate device memory.
 *
 * The pages describe nothing like this; it exists for callers that cannot give the library
 * a workspace: a plugin inside a host program that owns all device memory and offers no
 * allocator, a serving loop that must not call cudaMalloc/cudaFree because they can
 * synchronise the device, or a caller whose device memory budget is fixed in advance.
 *
 * It runs the CUDA-core attention kernel (TV_PATH_AUTO or TV_PATH_SIMT; TV_PATH_TCGEN05
 * is rejected) and keeps the split-KV partial results in a fixed array of
 * TV_NOALLOC_SCRATCH_BYTES bytes that the library reserves in device memory on every GPU
 * that loads it, held until the process exits.  It never allocates.  The caller still
 * passes every input and output through `a`.
 *   - The first call on a device looks up the array's address on that device (a
 *     cudaGetSymbolAddress), whatever the request; so does the first call after the
 *     device's CUDA context changed (cudaDeviceReset, or another context made current),
 *     since the array then lives in a newly loaded module.  Make such a first call before
 *     any stream capture.
 *   - A request whose scratch need exceeds TV_NOALLOC_SCRATCH_BYTES returns
 *     TV_ERR_WORKSPACE with an explanation in tv_last_error().  The need is what
 *     tv_verify_attn_workspace_size(a) reports for the same arguments with
 *     a->path = TV_PATH_SIMT (with TV_PATH_AUTO on a tensor-core shape that query reports
 *     the tensor-core path's size instead).
 *   - All calls share the one array and it keeps the last call's contents (nothing in it
 *     needs to start at zero).  Calls whose kernels can overlap on the GPU -- unordered
 *     streams, several host threads -- race on it; the caller must serialise them.
 * Results equal tv_verify_attn's on the CUDA-core path.
 */
#define TV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int tv_verify_attn_noalloc(const tv_attn_args* a, void* stream);

/* Size in bytes of the fixed scratch array behind tv_verify_attn_noalloc. */
size_t tv_noalloc_scratch_bytes(void);

/*
 * tv_verify_prologue -- the steps before tv_verify_attn in one launch.
 *
 * [RoPE] §"The Thinking Process": cos/sin are computed once and reused; [RoPE] §"The
 * Broader Context: A Full Native Engine from Scratch": the engine manages the KV cache;
 * [VERIFY] §Context: the visibility mask.  Same results, bit for bit, as
 *     tv_build_visibility(parent -> anc, depth)
 *     tv_rope_neox(q_pe_in -> q_pe_out, position prefix_len + depth)
 *     tv_rope_neox(kpe_tree -> k_pe cache slots prefix_len + i)
 * plus the copy of the draft tokens' latent rows ckv_tree[b,i,:] into c_kv cache slot
 * prefix_len[b] + i, with each node's cos/sin computed once for all of them.
 */
typedef struct {
  uint32_t struct_size;      /* sizeof(tv_prologue_args): ABI check */
  int32_t B, Q, H;           /* Q <= 64 (tree) */
  int32_t d_latent, d_rope;  /* d_rope % 8 == 0, d_rope <= 512, H * d_rope <= 8192;
                                d_latent % 8 == 0 */
  const int32_t* parent;     /* device [B, Q] draft tree */
  const int32_t* prefix_len; /* device [B] */
  const void* q_pe_in;       /* device [B, Q, H, d_rope] contiguous, q_dt */
  void* q_pe_out;            /* same shape and type; may equal q_pe_in */
  tv_dtype q_dt;
  const void* kpe_tree;      /* device [B, Q, d_rope] un-rotated draft keys, kv_dt */
  const void* ckv_tree;      /* device [B, Q, d_latent] draft latent rows, kv_dt; nullable */
  void* c_kv;                /* cache arrays (kv_dt), rows 16-byte aligned */
  void* k_pe;
  tv_dtype kv_dt;
  int64_t ckv_row_stride, kpe_row_stride; /* elements */
  tv_cache_layout cache;     /* slots outside it (or beyond num_rows when set) are skipped */
  uint64_t* anc;             /* device [B, Q] out */
  int32_t* depth;            /* device [B, Q] out */
  double rope_base;
  int32_t* status;           /* device int32, nullable: TV_ERR_INVALID_TREE for a bad tree
                                (that sequence's rows are left alone) */
} tv_prologue_args;

int tv_verify_prologue(const tv_prologue_args* a, void* stream);

/*
 * tv_build_tree -- best-first draft-tree construction under a node budget.
 *
 * [VERIFY] §"The Context: What Led to This Moment": the engine's GPU best-first tree
 * builder replaces a per-request CPU heapq implementation.  The pages give no formula; the
 * reading taken here: the drafter proposes, for each depth d = 1..L after the root, K
 * candidate tokens with log-probabilities sorted in descending order (one list per depth,
 * shared by every path).  A node is a path of candidate ranks (r_1..r_d) with token
 * cand_tokens[b,d-1,r_d] and score lp[b,0,r_1] + ... + lp[b,d-1,r_d] (float32, added in
 * depth order).  The tree is the root plus the `budget` best nodes taken best first --
 * larger score, then smaller depth, then lexicographically smaller rank path -- numbered
 * in the order taken (node 0 is the root), so parent[i] < i.
 *
 * logprobs    : device [B, L, K] float32, finite, descending over K (a sequence whose
 *               lists are not sorted gets TV_ERR_INVALID_ARG in *status).
 * cand_tokens : device [B, L, K] int32.
 * root_token  : device [B] int32, nullable (node 0's token; -1 when NULL).
 * parent, tokens : device [B, budget+1] int32 out, the tree as tv_build_visibility and
 *               tv_tree_accept take it.  depth [B, budget+1] int32 and score [B, budget+1]
 *               float32 are optional outputs (nullable).
 * Returns TV_ERR_UNSUPPORTED unless L <= 16, K <= 16, budget <= 63 (the verify kernels'
 * q_len <= 64), TV_ERR_INVALID_ARG for a budget above the number of possible nodes.
 */
int tv_build_tree(const float* logprobs, const int32_t* cand_tokens, const int32_t* root_token,
                  int B, int L, int K, int budget, int32_t* parent, int32_t* tokens,
                  int32_t* depth, float* score, int32_t* status, void* stream);

/*
 * tv_tree_accept -- greedy acceptance of a verified draft tree.
 *
 * [RoPE] §"The Broader Context: A Full Native Engine from Scratch" names a greedy
 * tree-accept kernel in the DDTree decode loop, whose greedy output must equal greedy
 * autoregressive decoding token for token; [GOLDEN] §"Context: The Quest for a
 * Hyper-Optimized Inference Stack" lists it among the engine's three custom kernels.  The
 * pages give no formula; the reading taken here:
 *   target[b,i] = argmax_v logits[b,i,v]  (the target model's next token after node i;
 *                 ties go to the smallest token id; logits must be finite),
 *   walk from the root: the next accepted node is the child c of the current node with
 *   tokens[b,c] == target[b,current] (the smallest such c), until there is none; the
 *   bonus token is target[b,last accepted node].
 *
 * logits     : device [B, Q, vocab] (row (b,i) at logits + (b*Q+i)*logits_row_stride
 *              elements), F32 or BF16 (rows at 16-byte boundaries stream fastest).
 * parent     : device [B, Q] int32 draft tree (as for tv_build_visibility).
 * tokens     : device [B, Q] int32 draft token of every node (node 0's entry, the root
 *              token, is not read).
 * target     : device [B, Q] int32 out, nullable: the argmax of every node's logits.
 * accept_len : device [B] int32 out: accepted draft nodes A (0 .. Q-1).
 * path       : device [B, Q] int32 out: 0 (the root), then the accepted nodes in depth
 *              order, then -1.
 * new_tokens : device [B, Q] int32 out: the accepted draft tokens, then the bonus token,
 *              then -1 (A + 1 tokens emitted by the step).
 * status     : see the conventions.  A sequence with an invalid parent array gets A = 0,
 *              path = [0, -1, ...], new_tokens all -1 and TV_ERR_INVALID_TREE.
 * workspace  : device memory of tv_tree_accept_workspace_size(B, Q, vocab) bytes, 256-byte
 *              aligned (the per-chunk argmax keys); scratch, reusable after the call.
 * Returns TV_ERR_UNSUPPORTED for Q > 64, TV_ERR_INVALID_ARG for bad sizes or pointers,
 * TV_ERR_WORKSPACE for a missing, misaligned or short workspace.
 */
size_t tv_tree_accept_workspace_size(int B, int Q, int64_t vocab);
int tv_tree_accept(const void* logits, tv_dtype logits_dt, int64_t vocab,
                   int64_t logits_row_stride, const int32_t* parent, const int32_t* tokens,
                   int B, int Q, int32_t* target, int32_t* accept_len, int32_t* path,
                   int32_t* new_tokens, int32_t* status, void* workspace, size_t ws_bytes,
                   void* stream);

/*
 * tv_compact_kv -- post-verify compaction of the latent KV cache.
 *
 * [RoPE] §"The Broader Context: A Full Native Engine from Scratch": the engine keeps a KV
 * cache with post-verify compaction.  Reading taken here: node i's row sits at logical key
 * prefix_len[b] + i; after acceptance the node at depth d (path[b, d], from tv_tree_accept)
 * moves to logical key prefix_len[b] + d, for d = 1 .. accept_len[b] (the root stays), so
 * that the accepted tokens follow the prefix contiguously.  Both the c_kv row and the k_pe
 * row move; the k_pe row was rotated at position prefix_len + depth, which is its new key
 * index, so it moves unchanged.  new_prefix_len[b] = prefix_len[b] + 1 + accept_len[b].
 *
 * c_kv, k_pe : device cache arrays (rows of d_latent / d_rope elements at the given row
 *              strides, in elements); row sizes, strides and pointers must be multiples of
 *              16 bytes.  Updated in place.
 * cache      : host struct, the cache geometry (page table or contiguous) with num_rows > 0.
 * prefix_len [B], path [B, Q], accept_len [B]: device int32 (path and accept_len as written
 *              by tv_tree_accept).  new_prefix_len [B]: device int32 out (may alias
 *              prefix_len only if the caller does not need the old value).
 * status     : a sequence whose path or keys fall outside the geometry is left unmoved,
 *              keeps new_prefix_len = prefix_len and gets TV_ERR_BOUNDS.
 */
int tv_compact_kv(void* c_kv, void* k_pe, tv_dtype kv_dt, int64_t ckv_row_stride,
                  int64_t kpe_row_stride, int d_latent, int d_rope,
                  const tv_cache_layout* cache, const int32_t* prefix_len, const int32_t* path,
                  const int32_t* accept_len, int B, int Q, int32_t* new_prefix_len,
                  int32_t* status, void* stream);

/* Text for a tv_status code (static storage). */
const char* tv_status_string(int code);

/* Description of the last failure on this host thread ("" if none). */
const char* tv_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int tv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TV_H_ */
