// k_attn_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) path of tv_verify_attn.
//
// Method: "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA
// Attention Kernel" (§Context, §"Input Knowledge Required") and "The Golden Reference: A
// Pivotal Moment in Building a Native DDTree Inference Engine" (§"The Absorb Form of
// MLA"): for every (node, head) row, softmax over the visible keys of
// scale*(q_latent.c_kv + q_pe.k_pe), then the softmax-weighted sum of c_kv rows.
//
// Shape of the work.  All H heads of all Q tree nodes of a sequence read the same latent
// KV rows, so the rows (node, head) of one sequence form the M dimension of two dense
// contractions: S = Q K^T (K = d_latent + d_rope = 576) and O = P V (N = d_latent = 512).
// A 128-row tile's fp32 O accumulator alone (128 x 512 x 4 B = 256 KB) fills an SM's
// tensor memory, leaving no room for S.  So each tile is served by a cluster of two CTAs
// on two SMs that split the two contractions between them:
//
//   rank 0 ("S side"): holds the tile's queries in TMEM (A operand of QK^T), receives each
//     64-key block's latent rows (two 3-D boxes of 4 chunks, loaded for it by rank 1's TMA
//     engine) and loads the rope chunk itself, computes S into one of two TMEM
//     buffers, runs the masked online softmax (lazy rescaling: the running max only moves
//     when it grows by more than 2^8), and ships each block's P (bf16, in the swizzled
//     K-major layout the MMA reads), the per-row rescale factors and, at the end, the row
//     sums to rank 1 with one bulk shared->shared copy per block.  It writes the lse.
//   rank 1 ("O side"): streams the same keys' latent chunks as the V operand (MN-major
//     B), accumulates O += P V in all 512 TMEM columns, applies the rare rescales, and at
//     the end of the tile normalises O by the row sums and writes it out.
//
// Per 64-key block the S side does 2*128*64*576 flops and the O side 2*128*512*64, so
// the pair is balanced to within 12%.  Warp roles per CTA (256 threads): warp 0 = TMA
// producer, warp 1 = MMA issuer (and TMEM allocator), warp 2 = message sender on rank 0
// and message bookkeeping on rank 1, warps 4-7 = the row-parallel math (thread = tile
// row, matching TMEM lanes).  Messages travel through 2 staging buffers on rank 0 and 4
// inbox buffers on rank 1, so the softmax never waits for the peer's round trip.
// Tiles are handed out round-robin to the persistent clusters; long KV ranges may be
// split across tiles and merged by the split combine kernel.
//
// Every wait is bounded (a wall-clock deadline); on expiry the kernel records
// TV_ERR_TIMEOUT, tells the peer CTA, drains its tensor-core work, frees its TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "sm100_ptx.h"
#include "tv_internal.h"

namespace tv {
namespace {

using namespace ptx;

constexpr int kDL = 512, kDR = 64, kBN = 64, kRows = 128;
constexpr int kChunkBytes = kBN * 128;          // 64 keys x 64 bf16
constexpr int kKChunks = 9;                     // 8 latent + 1 rope chunk per key block
constexpr int kHalf = 4 * kChunkBytes;          // 4 latent chunks: one 3-D TMA box
constexpr int kNLS = 5;                         // S-side latent ring stages (half key blocks)
constexpr int kNLO = 4;                         // O-side latent ring stages
constexpr int kNR = 2;                          // S-side rope ring stages
constexpr int kMsgAlpha = 16384, kMsgL = 16896, kMsgHdr = 17408, kMsgBytes = 17424;
constexpr int kMsgStride = 18432;
constexpr int kNStage = 2;                      // S-side staging buffers
constexpr int kNInbox = 4;                      // O-side inbox buffers
constexpr int kThreads = 256;
// Shared memory, from offset 0 in each CTA: its own latent ring (both are filled by rank
// 1's TMA engine: rank 0's through a multicast addressed to rank 0 only), then on rank 0
// the rope ring and the staging buffers, on rank 1 the inbox.
constexpr int kLatS = kNLS * kHalf;
constexpr int kLatO = kNLO * kHalf;
constexpr int kSideA = kLatS + kNR * kChunkBytes + kNStage * kMsgStride;
constexpr int kSideB = kLatO + kNInbox * kMsgStride;
constexpr int kSmemBytes = (kSideA > kSideB ? kSideA : kSideB) + 1024;
constexpr uint32_t kTmQ = 0, kTmS0 = 288, kTmS1 = 352;       // S-side TMEM columns
constexpr uint32_t kFlagFirst = 1, kFlagRescale = 2, kFlagFinal = 4;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);

struct TcParams {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_pe;
  const int32_t* page_table;
  int64_t kv_stride_b;
  const int32_t* prefix_len;
  const uint64_t* anc;
  float* out;
  float* lse;
  float* ws_out;
  float* ws_lse;
  int32_t* status;
  int64_t rows_total;  // B*Q*H
  int32_t max_pages;
  int32_t B, H, Q, max_prefix;
  int32_t tiles_per_seq, splits, chunk, n_items;
  int32_t paged;
  float scale_log2;
};

struct Shared {
  uint64_t slat_full[kNLS], slat_consumed[kNLS], slat_empty[kNLS];
  uint64_t olat_full[kNLO], olat_consumed[kNLO];
  uint64_t rope_full[kNR], rope_empty[kNR];
  uint64_t s_full[2], s_empty[2];
  uint64_t q_ready, q_free, msg_ready[kNStage], staging_free[kNStage], pdst_free[kNInbox];
  uint64_t p_full[kNInbox], p_consumed[kNInbox];
  uint64_t drain, job_full, corr_done, epi_done, final_bar;
  uint32_t tmem_base;
  volatile int abort;
  volatile int job_type, job_buf;
};

struct Item {
  int b, t, s, P, nb;
  int rot;  // first key block of this tile's sweep (see decode)
  int64_t k0;
  bool bad;
};

__device__ __noinline__ Item decode(const TcParams& p, int item) {
  Item it;
  it.t = item % p.tiles_per_seq;
  const int bs = item / p.tiles_per_seq;
  it.s = bs % p.splits;
  it.b = bs / p.splits;
  it.P = p.prefix_len[it.b];
  const int64_t kv_len = (int64_t)it.P + p.Q;
  it.bad = it.P < 0 || it.P > p.max_prefix ||
           (p.paged ? kv_len > (int64_t)p.max_pages * kBN : kv_len > p.kv_stride_b);
  it.k0 = (int64_t)it.s * p.chunk;
  int64_t k1 = it.k0 + p.chunk < kv_len ? it.k0 + p.chunk : kv_len;
  if (it.bad) k1 = it.k0;
  it.nb = k1 > it.k0 ? (int)((k1 - it.k0 + kBN - 1) / kBN) : 0;
  // The row tiles of one sequence run at the same time on neighbouring clusters; each
  // starts its sweep over the key blocks at a different block so that they do not all
  // request the same cache lines at once (the softmax is independent of block order).
  it.rot = it.nb > 0 ? (int)(((int64_t)it.t * it.nb) / p.tiles_per_seq) : 0;
  return it;
}

// Key block visited at step j of the tile's sweep.
__device__ __forceinline__ int sweep_block(const Item& it, int j) {
  const int jj = j + it.rot;
  return jj >= it.nb ? jj - it.nb : jj;
}

__device__ __forceinline__ void raise_abort(Shared& sh, int32_t* status, int code) {
  if (!sh.abort) {
    sh.abort = 1;
    report(status, code);
    // tell the peer CTA so that its waits end quickly too
    const uint32_t peer = map_to_rank(smem_u32((const void*)&sh.abort), cluster_rank() ^ 1u);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer), "r"(1) : "memory");
  }
}

// Bounded wait on phase `parity` of a local mbarrier: one inline probe, then an out-of-line
// polling loop with a wall-clock deadline (kept out of line to keep hot loops small).
__device__ __noinline__ bool wait_bar_slow(Shared& sh, uint32_t a, uint32_t parity,
                                           int32_t* status) {
  const uint64_t t0 = globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (sh.abort) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      raise_abort(sh, status, TV_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar(Shared& sh, uint64_t* bar, uint32_t parity,
                                         int32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  return wait_bar_slow(sh, a, parity, status);
}

__device__ __forceinline__ int64_t block_row0(const TcParams& p, const Item& it, int j) {
  const int64_t key0 = it.k0 + (int64_t)j * kBN;
  if (p.paged) return (int64_t)p.page_table[(int64_t)it.b * p.max_pages + key0 / kBN] * kBN;
  return (int64_t)it.b * p.kv_stride_b + key0;
}

// Visibility of keys key0 .. key0+63 for a row whose node has ancestor bitset `anc`: bit k
// set iff key0 + k < k1 and (key0 + k is a prefix key, or the tree node key0 + k - P is an
// ancestor-or-self of the row's node).
__device__ __forceinline__ uint64_t block_vis(int64_t key0, int64_t P, int64_t k1, uint64_t anc) {
  const int64_t np = P - key0;
  const uint64_t pm = np >= 64 ? ~0ull : (np <= 0 ? 0ull : ((1ull << np) - 1));
  const int64_t sh = key0 - P;
  const uint64_t tm = sh >= 0 ? (sh >= 64 ? 0ull : (anc >> sh)) : (-sh >= 64 ? 0ull : (anc << (-sh)));
  const int64_t nr = k1 - key0;
  const uint64_t rm = nr >= 64 ? ~0ull : (nr <= 0 ? 0ull : ((1ull << nr) - 1));
  return (pm | tm) & rm;
}

__device__ __forceinline__ float max64(const float* t) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = fmaxf(fmaxf(t[4 * i], t[4 * i + 1]), fmaxf(t[4 * i + 2], t[4 * i + 3]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] = fmaxf(a[i], a[i + w]);
  return a[0];
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ===================================================================================
// rank 0: QK^T + softmax
// ===================================================================================
__device__ void s_side(const TcParams& p, const CUtensorMap* map_ckv, const CUtensorMap* map_kpe,
                       Shared& sh, unsigned char* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* lat = smem;
  unsigned char* rope = smem + kLatS;
  unsigned char* stage = rope + kNR * kChunkBytes;
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer: the rope chunk of each key block ----------------
    // (the latent chunks arrive by multicast from rank 1's producer)
    if (lane == 0) {
      prefetch_tensormap(map_kpe);
      uint32_t kb = 0;
      for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
        const Item it = decode(p, item);
        // the page-table lookup for the next block is issued a block ahead
        int next_row = it.nb > 0 ? (int)block_row0(p, it, sweep_block(it, 0)) : 0;
        for (int j = 0; j < it.nb; ++j, ++kb) {
          const int row0 = next_row;
          if (j + 1 < it.nb) next_row = (int)block_row0(p, it, sweep_block(it, j + 1));
          const uint32_t st = kb % kNR;
          if (!wait_bar(sh, &sh.rope_empty[st], ((kb / kNR) & 1) ^ 1, p.status)) return;
          mbar_arrive_expect_tx(&sh.rope_full[st], kChunkBytes);
          tma_load_2d(rope + st * kChunkBytes, map_kpe, 0, row0, &sh.rope_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: S = Q K^T -----------------------------------------
    if (lane == 0) {
      uint32_t kb = 0, sc = 0, qc = 0;
      for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
        const Item it = decode(p, item);
        if (it.nb == 0) continue;
        if (!wait_bar(sh, &sh.q_ready, qc & 1, p.status)) break;
        ++qc;
        tc_fence_after();
        for (int j = 0; j < it.nb && !sh.abort; ++j, ++sc, ++kb) {
          const uint32_t sb = sc & 1;
          if (!wait_bar(sh, &sh.s_empty[sb], ((sc >> 1) & 1) ^ 1, p.status)) break;
          tc_fence_after();  // the softmax warps' TMEM reads of this S buffer come first
          const uint32_t d = tmem + (sb ? kTmS1 : kTmS0);
          bool ok = true;
          for (int h = 0; h < 2 && ok; ++h) {
            const uint32_t u = 2 * kb + h, st = u % kNLS;
            if (!wait_bar(sh, &sh.slat_full[st], (u / kNLS) & 1, p.status)) { ok = false; break; }
            const uint32_t sa = smem_u32(lat + st * kHalf);
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(d, tmem + kTmQ + 32 * (4 * h + c) + 8 * kk,
                       smem_desc(sa + c * kChunkBytes + 32 * kk, 16, 1024, 2), kIdescQK,
                       (h | c | kk) != 0);
            mma_commit(&sh.slat_consumed[st]);
          }
          const uint32_t rs = kb % kNR;
          if (!ok || !wait_bar(sh, &sh.rope_full[rs], (kb / kNR) & 1, p.status)) break;
          const uint32_t ra = smem_u32(rope + rs * kChunkBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(d, tmem + kTmQ + 32 * 8 + 8 * kk, smem_desc(ra + 32 * kk, 16, 1024, 2),
                   kIdescQK, 1);
          mma_commit(&sh.rope_empty[rs]);
          mma_commit(&sh.s_full[sb]);
        }
        mma_commit(&sh.q_free);
      }
      mma_commit(&sh.final_bar);
      wait_bar(sh, &sh.final_bar, 0, p.status);
    }
  } else if (warp == 3) {
    // ---------------- latent-ring helper: once this CTA has read a stage, re-arm it and
    // tell rank 1's producer for this ring that the stage may be refilled ---------------
    if (lane == 0) {
      const uint32_t peer = cluster_rank() ^ 1u;
      uint32_t u = 0;
      for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
        const Item it = decode(p, item);
        for (int j = 0; j < 2 * it.nb; ++j, ++u) {
          const uint32_t st = u % kNLS;
          if (!wait_bar(sh, &sh.slat_consumed[st], (u / kNLS) & 1, p.status)) return;
          mbar_arrive_expect_tx(&sh.slat_full[st], kHalf);
          mbar_arrive_remote(map_to_rank(smem_u32(&sh.slat_empty[st]), peer));
        }
      }
    }
  } else if (warp == 2) {
    // ---------------- sender: staging buffer -> peer inbox, one bulk copy per block --
    const uint32_t peer = cluster_rank() ^ 1u;
    unsigned char* peer_inbox_local = smem + kLatO;  // same offset in the peer
    uint32_t mc = 0;
    bool live = true;
    for (int item = cid; item < p.n_items && live && !sh.abort; item += ncl) {
      const Item it = decode(p, item);
      for (int j = 0; j < it.nb; ++j, ++mc) {
        const uint32_t sbuf = mc % kNStage, ib = mc % kNInbox;
        if (!__all_sync(0xffffffffu, wait_bar(sh, &sh.msg_ready[sbuf], (mc / kNStage) & 1, p.status))) {
          live = false;
          break;
        }
        unsigned char* msg = stage + sbuf * kMsgStride;
        const float* alpha = reinterpret_cast<const float*>(msg + kMsgAlpha);
        bool resc = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) resc |= alpha[lane * 4 + q] != 1.f;
        resc = __any_sync(0xffffffffu, resc);
        if (lane == 0) {
          const uint32_t flags = (j == 0 ? kFlagFirst : 0u) | (j == it.nb - 1 ? kFlagFinal : 0u) |
                                 ((resc && j > 0) ? kFlagRescale : 0u);
          *reinterpret_cast<volatile uint32_t*>(msg + kMsgHdr) = flags;
          fence_proxy_async_smem();
          if (wait_bar(sh, &sh.pdst_free[ib], ((mc / kNInbox) & 1) ^ 1, p.status)) {
            const uint32_t dst = map_to_rank(smem_u32(peer_inbox_local + ib * kMsgStride), peer);
            const uint32_t bar = map_to_rank(smem_u32(&sh.p_full[ib]), peer);
            bulk_copy_to_cluster(dst, msg, kMsgBytes, bar);
            bulk_commit();
            bulk_wait_read<0>();
          }
          mbar_arrive(&sh.staging_free[sbuf]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  } else if (warp >= 4) {
    // ---------------- softmax warpgroup: thread r owns tile row r ------------------
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    uint32_t sc = 0, qc = 0, mc = 0;
    for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
      const Item it = decode(p, item);
      const int trow = it.t * kRows + r;
      const bool vrow = trow < p.Q * p.H;
      const int64_t grow = (int64_t)it.b * p.Q * p.H + trow;
      float* lse_dst = p.splits == 1 ? p.lse + grow : p.ws_lse + (int64_t)it.s * p.rows_total + grow;
      if (it.bad && r == 0 && it.t == 0 && it.s == 0) report(p.status, TV_ERR_BOUNDS);
      if (it.nb == 0) {
        if (vrow) *lse_dst = -INFINITY;
        continue;
      }
      {
        // warm L2 with the next tile's queries while this tile runs
        const int nxt = item + ncl;
        if (nxt < p.n_items) {
          const Item in = decode(p, nxt);
          const int nrow = in.t * kRows + r;
          if (in.nb > 0 && nrow < p.Q * p.H) {
            const int64_t ng = (int64_t)in.b * p.Q * p.H + nrow;
            const char* qlp = reinterpret_cast<const char*>(p.q_latent + ng * kDL);
#pragma unroll
            for (int l128 = 0; l128 < 8; ++l128) prefetch_l2(qlp + 128 * l128);
            prefetch_l2(p.q_pe + ng * kDR);
          }
        }
      }
      const uint64_t anc = vrow ? p.anc[(int64_t)it.b * p.Q + trow / p.H] : 0ull;
      const int64_t kv_end = (int64_t)it.P + p.Q;
      const int64_t k1 = it.k0 + p.chunk < kv_end ? it.k0 + p.chunk : kv_end;

      // ---- queries of this row into TMEM columns [0, 288) ----
      // (each warp agrees on the outcome of a wait before its warp-collective TMEM ops)
      if (!__all_sync(0xffffffffu, wait_bar(sh, &sh.q_free, (qc & 1) ^ 1, p.status))) break;
      ++qc;
      tc_fence_after();
      {
        const uint4* ql = reinterpret_cast<const uint4*>(p.q_latent + grow * kDL);
        const uint4* qr = reinterpret_cast<const uint4*>(p.q_pe + grow * kDR);
#pragma unroll 1
        for (int c0 = 0; c0 < kKChunks; c0 += 3) {
          uint32_t w[3][32];
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) {
            const int ch = c0 + cc;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              uint4 v = make_uint4(0, 0, 0, 0);
              if (vrow) v = ch < 8 ? __ldg(ql + 8 * ch + e) : __ldg(qr + e);
              w[cc][4 * e + 0] = v.x;
              w[cc][4 * e + 1] = v.y;
              w[cc][4 * e + 2] = v.z;
              w[cc][4 * e + 3] = v.w;
            }
          }
          __syncwarp();
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) tmem_st32(tmem + lane_base + kTmQ + 32 * (c0 + cc), w[cc]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sh.q_ready);

      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.nb; ++j, ++sc, ++mc) {
        const uint32_t sb = sc & 1;
        if (!__all_sync(0xffffffffu, wait_bar(sh, &sh.s_full[sb], (sc >> 1) & 1, p.status))) break;
        tc_fence_after();
        float t[64];
        {
          uint32_t sr[64];
          tmem_ld32(tmem + lane_base + (sb ? kTmS1 : kTmS0), sr);
          tmem_ld32(tmem + lane_base + (sb ? kTmS1 : kTmS0) + 32, sr + 32);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&sh.s_empty[sb]);
#pragma unroll
          for (int k = 0; k < 64; ++k) t[k] = __uint_as_float(sr[k]);
        }
        const int64_t key0 = it.k0 + (int64_t)sweep_block(it, j) * kBN;
        const uint64_t vis =
            (key0 + kBN > it.P || key0 + kBN > k1) ? block_vis(key0, it.P, k1, anc) : ~0ull;

        // t = score*c - m (masked keys -inf), exponentiated against the current running
        // max while the block max is reduced alongside; only a max that grew by more than
        // 2^8 (rare) sends the block through a second pass.  A row's first visible keys
        // (m = -inf) take the second pass too: their max is not known in advance.
        const float mref = m == -INFINITY ? 0.f : m;
#pragma unroll
        for (int k = 0; k < 64; ++k) t[k] = ((vis >> k) & 1ull) ? fmaf(t[k], c, -mref) : -INFINITY;
        uint32_t pk[32];
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          const float p0 = ex2(t[k]), p1 = ex2(t[k + 1]);
          s4[(k >> 1) & 3] += p0 + p1;
          pk[k >> 1] = pack_bf16(p0, p1);
        }
        const float bmt = max64(t);  // block max relative to mref
        float alpha = 1.f;
        if (bmt > (m == -INFINITY ? -INFINITY : kRescaleThreshold)) {
          if (l > 0.f) alpha = ex2(-bmt);
          m = mref + bmt;
          s4[0] = s4[1] = s4[2] = s4[3] = 0.f;
#pragma unroll
          for (int k = 0; k < 64; k += 2) {
            const float p0 = ex2(t[k] - bmt), p1 = ex2(t[k + 1] - bmt);
            s4[(k >> 1) & 3] += p0 + p1;
            pk[k >> 1] = pack_bf16(p0, p1);
          }
        }
        const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        l = l * alpha + sum;

        // ---- P (bf16, swizzled K-major), alpha and, last, the row sum into staging ----
        const uint32_t sbuf = mc % kNStage;
        if (!__all_sync(0xffffffffu,
                        wait_bar(sh, &sh.staging_free[sbuf], ((mc / kNStage) & 1) ^ 1, p.status)))
          break;
        unsigned char* msg = stage + sbuf * kMsgStride;
        unsigned char* rowp = msg + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(rowp + ((q ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        reinterpret_cast<float*>(msg + kMsgAlpha)[r] = alpha;
        if (j == it.nb - 1) reinterpret_cast<float*>(msg + kMsgL)[r] = l;
        fence_proxy_async_smem();
        mbar_arrive(&sh.msg_ready[sbuf]);
      }
      if (vrow && !sh.abort)
        *lse_dst = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

// ===================================================================================
// rank 1: O += P V, rescale, epilogue
// ===================================================================================
__device__ void o_side(const TcParams& p, const CUtensorMap* map_ckv, Shared& sh,
                       unsigned char* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* lat = smem;
  unsigned char* inbox = smem + kLatO;
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer for rank 0's latent ring (multicast addressed to rank
    // 0 only, so this CTA's engine serves both rings) ----------------------------------
    if (lane == 0) {
      prefetch_tensormap(map_ckv);
      uint32_t u = 0;
      for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
        const Item it = decode(p, item);
        int next_row = it.nb > 0 ? (int)block_row0(p, it, sweep_block(it, 0)) : 0;
        for (int j = 0; j < it.nb; ++j) {
          const int row0 = next_row;
          if (j + 1 < it.nb) next_row = (int)block_row0(p, it, sweep_block(it, j + 1));
          for (int h = 0; h < 2; ++h, ++u) {
            const uint32_t st = u % kNLS;
            // rank 0 has read the stage's previous fill and re-armed its barrier
            if (!wait_bar(sh, &sh.slat_empty[st], ((u / kNLS) & 1) ^ 1, p.status)) return;
            tma_load_3d_multicast(lat + st * kHalf, map_ckv, 0, row0, 4 * h, &sh.slat_full[st],
                                  (uint16_t)0x1);
          }
        }
      }
    }
  } else if (warp == 3) {
    // ---------------- TMA producer for this CTA's latent ring ---------------------------
    if (lane == 0) {
      prefetch_tensormap(map_ckv);
      uint32_t u = 0;
      for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
        const Item it = decode(p, item);
        int next_row = it.nb > 0 ? (int)block_row0(p, it, sweep_block(it, 0)) : 0;
        for (int j = 0; j < it.nb; ++j) {
          const int row0 = next_row;
          if (j + 1 < it.nb) next_row = (int)block_row0(p, it, sweep_block(it, j + 1));
          for (int h = 0; h < 2; ++h, ++u) {
            const uint32_t st = u % kNLO;
            if (!wait_bar(sh, &sh.olat_consumed[st], ((u / kNLO) & 1) ^ 1, p.status)) return;
            mbar_arrive_expect_tx(&sh.olat_full[st], kHalf);
            tma_load_3d(lat + st * kHalf, map_ckv, 0, row0, 4 * h, &sh.olat_full[st]);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: O += P V ------------------------------------------
    if (lane == 0) {
      uint32_t vc = 0, mc = 0, ic = 0, dc = 0, cc = 0;
      for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
        const Item it = decode(p, item);
        if (it.nb == 0) continue;
        if (ic > 0 && !wait_bar(sh, &sh.epi_done, (ic - 1) & 1, p.status)) break;
        tc_fence_after();
        uint32_t last_pb = 0;
        bool ok = true;
        for (int j = 0; j < it.nb && ok; ++j, ++mc) {
          const uint32_t pb = mc % kNInbox;
          last_pb = pb;
          if (!wait_bar(sh, &sh.p_full[pb], (mc / kNInbox) & 1, p.status)) { ok = false; break; }
          const uint32_t flags =
              *reinterpret_cast<volatile uint32_t*>(inbox + pb * kMsgStride + kMsgHdr);
          if (flags & kFlagRescale) {
            mma_commit(&sh.drain);
            if (!wait_bar(sh, &sh.drain, dc & 1, p.status)) { ok = false; break; }
            ++dc;
            sh.job_type = 1;
            sh.job_buf = (int)pb;
            mbar_arrive(&sh.job_full);
            if (!wait_bar(sh, &sh.corr_done, cc & 1, p.status)) { ok = false; break; }
            ++cc;
            tc_fence_after();
          }
          const uint32_t pa = smem_u32(inbox + pb * kMsgStride);
          for (int h = 0; h < 2; ++h, ++vc) {
            const uint32_t st = vc % kNLO;
            if (!wait_bar(sh, &sh.olat_full[st], (vc / kNLO) & 1, p.status)) { ok = false; break; }
            const uint32_t va = smem_u32(lat + st * kHalf);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + 256 * h, smem_desc(pa + 32 * kk, 16, 1024, 2),
                     smem_desc(va + 2048 * kk, 8192, 1024, 2), kIdescPV, (j | kk) != 0);
            mma_commit(&sh.olat_consumed[st]);
          }
          mma_commit(&sh.p_consumed[pb]);
        }
        if (!ok) break;
        mma_commit(&sh.drain);
        if (!wait_bar(sh, &sh.drain, dc & 1, p.status)) break;
        ++dc;
        sh.job_type = 2;
        sh.job_buf = (int)last_pb;
        mbar_arrive(&sh.job_full);
        ++ic;
      }
      if (!sh.abort && ic > 0) wait_bar(sh, &sh.epi_done, (ic - 1) & 1, p.status);
      sh.job_type = 0;  // exit
      mbar_arrive(&sh.job_full);
      mma_commit(&sh.final_bar);
      wait_bar(sh, &sh.final_bar, 0, p.status);
    }
  } else if (warp == 2) {
    // ---------------- inbox bookkeeping: re-arm and hand buffers back ---------------
    if (lane == 0) {
      const uint32_t peer = cluster_rank() ^ 1u;
      uint32_t mc = 0, ic = 0;
      for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
        const Item it = decode(p, item);
        if (it.nb == 0) continue;
        for (int j = 0; j < it.nb; ++j, ++mc) {
          const uint32_t pb = mc % kNInbox;
          if (!wait_bar(sh, &sh.p_consumed[pb], (mc / kNInbox) & 1, p.status)) return;
          if (j == it.nb - 1 && !wait_bar(sh, &sh.epi_done, ic & 1, p.status)) return;
          mbar_arrive_expect_tx(&sh.p_full[pb], kMsgBytes);
          mbar_arrive_remote(map_to_rank(smem_u32(&sh.pdst_free[pb]), peer));
        }
        ++ic;
      }
    }
  } else if (warp >= 4) {
    // ---------------- rescale / epilogue warpgroup: thread r owns tile row r -------
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    uint32_t jc = 0;
    for (int item = cid; item < p.n_items && !sh.abort; item += ncl) {
      const Item it = decode(p, item);
      const int trow = it.t * kRows + r;
      const bool vrow = trow < p.Q * p.H;
      const int64_t grow = (int64_t)it.b * p.Q * p.H + trow;
      float* dst = p.splits == 1 ? p.out + grow * kDL
                                 : p.ws_out + ((int64_t)it.s * p.rows_total + grow) * kDL;
      if (it.nb == 0) {
        if (vrow)
          for (int c = 0; c < kDL / 4; ++c)
            reinterpret_cast<float4*>(dst)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      for (;;) {
        // the four warps work on disjoint TMEM lanes; each warp agrees on the outcome
        if (!__all_sync(0xffffffffu, wait_bar(sh, &sh.job_full, jc & 1, p.status))) return;
        ++jc;
        const int type = sh.job_type, pb = sh.job_buf;
        tc_fence_after();
        if (type == 1) {
          const float alpha = reinterpret_cast<const float*>(inbox + pb * kMsgStride + kMsgAlpha)[r];
          // warp-uniform decision: the TMEM loads and stores below are warp-collective
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < 16; ++c) {
              uint32_t v[32];
              __syncwarp();
              tmem_ld32(tmem + lane_base + 32 * c, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              tmem_st32(tmem + lane_base + 32 * c, v);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(&sh.corr_done);
        } else if (type == 2) {
          const float lr = reinterpret_cast<const float*>(inbox + pb * kMsgStride + kMsgL)[r];
          const float inv = lr > 0.f ? 1.f / lr : 0.f;
#pragma unroll 1
          for (int c = 0; c < 16; ++c) {
            uint32_t v[32];
            __syncwarp();
            tmem_ld32(tmem + lane_base + 32 * c, v);
            tmem_wait_ld();
            if (vrow) {
              float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                d4[e] = make_float4(__uint_as_float(v[4 * e]) * inv, __uint_as_float(v[4 * e + 1]) * inv,
                                    __uint_as_float(v[4 * e + 2]) * inv, __uint_as_float(v[4 * e + 3]) * inv);
            }
          }
          tc_fence_before();
          mbar_arrive(&sh.epi_done);
          break;
        } else {
          return;  // exit job (only after an abort)
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap map_ckv,
               const __grid_constant__ CUtensorMap map_kpe) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ Shared sh;
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNLS; ++i) {
      mbar_init(&sh.slat_full[i], 1);
      mbar_init(&sh.slat_consumed[i], 1);
      mbar_init(&sh.slat_empty[i], 1);
    }
    for (int i = 0; i < kNLO; ++i) {
      mbar_init(&sh.olat_full[i], 1);
      mbar_init(&sh.olat_consumed[i], 1);
    }
    for (int i = 0; i < kNR; ++i) {
      mbar_init(&sh.rope_full[i], 1);
      mbar_init(&sh.rope_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.s_empty[i], 128);
    }
    for (int i = 0; i < kNStage; ++i) {
      mbar_init(&sh.msg_ready[i], 128);
      mbar_init(&sh.staging_free[i], 1);
    }
    for (int i = 0; i < kNInbox; ++i) {
      mbar_init(&sh.pdst_free[i], 1);
      mbar_init(&sh.p_full[i], 1);
      mbar_init(&sh.p_consumed[i], 1);
    }
    mbar_init(&sh.q_ready, 128);
    mbar_init(&sh.q_free, 1);
    mbar_init(&sh.drain, 1);
    mbar_init(&sh.job_full, 1);
    mbar_init(&sh.corr_done, 128);
    mbar_init(&sh.epi_done, 128);
    mbar_init(&sh.final_bar, 1);
    sh.abort = 0;
    sh.job_type = 0;
    sh.job_buf = 0;
    if (rank == 0) {
      // rank 0's latent stages start armed for their first fill (issued by rank 1)
      for (int i = 0; i < kNLS; ++i) mbar_arrive_expect_tx(&sh.slat_full[i], kHalf);
    }
    if (rank == 1) {
      // every inbox buffer starts armed for its first message
      for (int i = 0; i < kNInbox; ++i) mbar_arrive_expect_tx(&sh.p_full[i], kMsgBytes);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // barriers of both CTAs exist before any remote arrive or copy

  if (rank == 0)
    s_side(p, &map_ckv, &map_kpe, sh, smem);
  else
    o_side(p, &map_ckv, sh, smem);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(sh.tmem_base, 512);
  cluster_sync();  // neither CTA leaves while the other may still touch its memory
}

// ---- host side -----------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
int g_max_clusters[64] = {};
std::mutex g_mu;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Latent rows viewed as [64 elements][rows][8 chunks of 64 elements]: one box is 4 chunks
// of 64 rows, landing chunk-major in shared memory as four 128-byte-swizzled 8 KB tiles.
bool make_map_latent(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes) {
  cuuint64_t dims[3] = {64, rows, kDL / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, 64, 4};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
              uint64_t row_bytes) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int max_clusters() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_max_clusters[dev] == 0) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      int sms = current_sm_count();
      n = sms / 2;
    }
    g_max_clusters[dev] = n;
  }
  return g_max_clusters[dev];
}

}  // namespace

bool tc_supported(const tv_attn_args* a) {
  return a->q_dt == TV_BF16 && a->kv_dt == TV_BF16 && a->d_latent == kDL && a->d_rope == kDR &&
         a->cache.num_rows > 0 && a->cache.num_rows < (1ll << 31) &&
         (a->cache.page_table == nullptr || a->cache.page_size == kBN);
}

TcPlan tc_plan(const tv_attn_args* a) {
  TcPlan p{};
  const int clusters = max_clusters() > 0 ? max_clusters() : 74;
  p.clusters = clusters;
  p.tiles_per_seq = (a->Q * a->H + kRows - 1) / kRows;
  const int64_t tiles = (int64_t)a->B * p.tiles_per_seq;
  const int64_t kv_max = (int64_t)a->max_prefix_len + a->Q;
  int splits = a->num_splits;
  if (splits <= 0) {
    splits = 1;
    if (tiles < 2LL * clusters) {
      const int64_t want = (2LL * clusters + tiles - 1) / std::max<int64_t>(tiles, 1);
      const int64_t cap = std::max<int64_t>(1, kv_max / 512);
      splits = (int)std::max<int64_t>(1, std::min(want, cap));
    }
  }
  int64_t chunk = (kv_max + splits - 1) / splits;
  chunk = (chunk + kBN - 1) / kBN * kBN;
  if (chunk < kBN) chunk = kBN;
  p.chunk = (int)chunk;
  p.splits = (int)((kv_max + chunk - 1) / chunk);
  if (p.splits < 1) p.splits = 1;
  p.n_items = (int)(tiles * p.splits);
  return p;
}

size_t tc_workspace(const tv_attn_args* a, const TcPlan& p) {
  if (p.splits <= 1) return 0;
  const size_t rows = (size_t)a->B * a->Q * a->H;
  const size_t out_b = ((size_t)p.splits * rows * a->d_latent * 4 + 255) / 256 * 256;
  const size_t lse_b = ((size_t)p.splits * rows * 4 + 255) / 256 * 256;
  return out_b + lse_b;
}

cudaError_t launch_attn_tc(const tv_attn_args* a, const TcPlan& pl, void* ws, cudaStream_t st) {
  if (!get_encode()) return cudaErrorNotSupported;
  if (max_clusters() <= 0) return cudaErrorNotSupported;
  CUtensorMap mc, mk;
  if (!make_map_latent(&mc, a->c_kv, (uint64_t)a->cache.num_rows, (uint64_t)a->ckv_row_stride * 2))
    return cudaErrorInvalidValue;
  if (!make_map(&mk, a->k_pe, kDR, (uint64_t)a->cache.num_rows, (uint64_t)a->kpe_row_stride * 2))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.q_latent = (const __nv_bfloat16*)a->q_latent;
  p.q_pe = (const __nv_bfloat16*)a->q_pe;
  p.page_table = a->cache.page_table;
  p.kv_stride_b = a->cache.kv_stride_b;
  p.prefix_len = a->prefix_len;
  p.anc = a->anc;
  p.out = a->out;
  p.lse = a->lse;
  const size_t rows = (size_t)a->B * a->Q * a->H;
  p.ws_out = (float*)ws;
  p.ws_lse = ws ? (float*)((char*)ws + ((size_t)pl.splits * rows * a->d_latent * 4 + 255) / 256 * 256)
                : nullptr;
  p.status = a->status;
  p.rows_total = (int64_t)rows;
  p.max_pages = a->cache.max_pages;
  p.B = a->B;
  p.H = a->H;
  p.Q = a->Q;
  p.max_prefix = a->max_prefix_len;
  p.tiles_per_seq = pl.tiles_per_seq;
  p.splits = pl.splits;
  p.chunk = pl.chunk;
  p.n_items = pl.n_items;
  p.paged = a->cache.page_table != nullptr;
  p.scale_log2 = (float)((double)a->scale * 1.4426950408889634);
  if (p.n_items == 0) return cudaSuccess;

  const int ncl = std::min(pl.clusters, pl.n_items);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ncl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tc_kernel, p, mc, mk);
  if (e != cudaSuccess || pl.splits == 1) return e;
  return launch_combine(p.ws_out, p.ws_lse, pl.splits, (int64_t)rows, a->d_latent, a->out,
                        a->lse, st);
}

}  // namespace tv
