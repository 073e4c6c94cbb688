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
//   rank 0 ("S side"): holds the tile's latent queries in TMEM (A operand of QK^T) and
//     their rope part in shared memory, loads the keys 128 at a time (four 3-D boxes of
//     2 latent chunks and one rope box), computes S for 128 keys into one of two TMEM
//     buffers with N = 128 MMAs, runs the masked online softmax (lazy rescaling: the
//     running max only moves when a block's max exceeds it by more than 2^8), and writes
//     each 64-key half's P (bf16, in the swizzled K-major layout the MMA reads), the per-row
//     rescale factor and running row sum into a local staging buffer, which one thread
//     ships to rank 1's inbox with a bulk shared->shared copy (the copy engine streams it
//     while the softmax goes on; cluster shared-memory traffic runs at only about 21 bytes
//     per clock, so the softmax threads must not wait on it).  It writes the lse.
//   rank 1 ("O side"): streams each 64-key block's latent chunks as the V operand
//     (MN-major B), accumulates O += P V in all 512 TMEM columns, applies the rare
//     rescales, and at the end of the tile normalises O by the row sums and writes it out.
//
// Per 128 keys the S side issues 36 MMAs of 128x128x16 and the O side 16 of 128x256x16,
// so the pair is balanced to within 12%.  Warp roles per CTA (256 threads): warp 0 = TMA
// producer, warp 1 = MMA issuer (and TMEM allocator), warps 4-7 = the row-parallel math
// (thread = tile row, matching TMEM lanes; on rank 0 thread 0 of them also issues the
// message copies); warps 2-3 idle.
//
// Keys come from a row-major view (c_kv row, k_pe row per key); a 128-key step of such a
// view is one box of 128 consecutive rows.  A contiguous cache is that view.  A paged
// cache keeps 64-key pages in any order; by default every 128-key step of every sequence
// gets its own tensor maps, built by prep_kernel -- a 5-D view {64 elements, 8 rows, 8 row
// groups, 2 pages, chunks} whose page dimension strides from the step's lower page to its
// other page, so that one box lands both pages' rows in the 128-row layout the MMA reads.
// If the step's second page lies below its first, the view starts at the lower one and S
// comes out with its two halves swapped, which the softmax undoes.  On request
// (TV_PAGED_GATHER) gather_kv_kernel first copies the pages into a contiguous view in the
// workspace instead.
//
// The schedule (computed by prep_kernel on the device from the prefix lengths): whole
// 128-row tiles are dealt to the persistent clusters longest first in rounds, the last
// rounds to the least-loaded clusters; the tiles left over are cut into pieces of about
// equal length, at most one piece per cluster.  The pieces of a split tile write partial
// results that merge_kernel combines.
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
#include "tv_testing.h"

namespace tv {
namespace {

using namespace ptx;

constexpr int kDL = 512, kDR = 64, kBN = 64, kStep = 128, kRows = 128;
constexpr int kChunkS = kStep * 128;            // 128 keys x 64 bf16 (S side)
constexpr int kStageS = 2 * kChunkS;            // 2 latent chunks: one 3-D box
constexpr int kNLS = 5;                         // S-side latent ring stages
constexpr int kNRope = 1;                       // S-side rope stages
constexpr int kChunkO = kBN * 128;              // 64 keys x 64 bf16 (O side)
constexpr int kHalfO = 4 * kChunkO;             // 4 latent chunks of a 64-key block
constexpr int kNLO = 4;                         // O-side latent ring stages
// A message carries one 64-key block: P (128 rows x 64 keys bf16), then per row the
// rescale factor and running row sum (fp32), then one flags word padded to 16 bytes.
constexpr int kMsgAlpha = 16384, kMsgL = 16896, kMsgFlags = 17408;
constexpr uint32_t kMsgBytes = 17424;
constexpr int kMsgStride = 18432;               // inbox buffers (P 1024-byte aligned)
constexpr int kNInbox = 4;
constexpr int kNStg = 2;                        // S-side staging buffers (one step)
constexpr int kThreads = 256;
// Shared memory, from offset 0 in each CTA.  Rank 0: latent ring, rope stages, the tile's
// rope queries, staging.  Rank 1: latent ring, inbox.
constexpr int kRopeOff = kNLS * kStageS;
constexpr int kQropeOff = kRopeOff + kNRope * kChunkS;
constexpr int kStgOff = kQropeOff + kRows * 128;
constexpr int kSideA = kStgOff + kNStg * (int)kMsgBytes;
constexpr int kInboxOff = kNLO * kHalfO;
constexpr int kSideB = kInboxOff + kNInbox * kMsgStride;
constexpr int kSideMax = kSideA > kSideB ? kSideA : kSideB;
// O side: the epilogue's staging chunks (4 warps x 32 rows x 32 fp32) after the inbox
constexpr int kEpiOff = kSideB;
static_assert(kEpiOff + 4 * 32 * 32 * 4 <= kSideMax, "epilogue staging must fit");

constexpr uint32_t kTmQ = 0, kTmS0 = 256, kTmS1 = 384;       // S-side TMEM columns
constexpr uint32_t kFlagRescale = 2;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // deadline of every wait (wall clock)
constexpr uint64_t kDrainNs = 2000000000ull;    // deadline of the exit drains
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);

struct TcParams {
  const __nv_bfloat16* q_latent;
  const __nv_bfloat16* q_pe;
  int64_t seq_rows;  // contiguous cache: rows between consecutive sequences
  int64_t seq_cap;   // longest KV a sequence may have
  const CUtensorMap* step_maps;  // paged cache: [B][steps_per_seq][latent, rope] maps
  const uint8_t* step_swap;      // paged cache: 1 where a step's pages come in swapped
  const int32_t* page_table;
  int32_t steps_per_seq, max_pages, paged;
  const int32_t* prefix_len;
  const uint64_t* anc;
  float* out;
  float* lse;
  float* ws_out;       // partial outputs of split tiles: [slot][128 rows][512]
  float* ws_lse;       // their log-sum-exps: [slot][128 rows]

  int32_t* status;
  int64_t rows_total;  // B*Q*H
  int32_t B, H, Q, max_prefix;
  int32_t tiles_per_seq;
  const int4* items;     // per work item two records: {b, t, s0, s1}, {P, pieces, slot, base}
  const int32_t* cl_start;  // cluster c takes items cl_start[c] .. cl_start[c+1]-1
  float scale_log2;
  uint64_t timeout_ns;        // deadline of every wait
  int32_t causal;             // TV_MASK_CAUSAL: row (node i, head) sees keys 0 .. P + i
  int32_t test_skip_loads;    // testing hook: the S-side producer issues no key loads
  int32_t* test_exit_counts;  // testing hook: [CTAs that left, CTAs that left aborted]
};

struct Shared {
  uint64_t slat_full[kNLS], slat_empty[kNLS];
  uint64_t olat_full[kNLO], olat_empty[kNLO];
  uint64_t rope_full[kNRope], rope_empty[kNRope];
  uint64_t s_full[2], s_empty[2];
  uint64_t qr_full, q_free, pdst_free[kNInbox];
  uint64_t p_full[kNInbox];
  uint64_t drain, job_full, corr_done, epi_done, final_bar;
  uint64_t timeout_ns;
  uint32_t tmem_base;
  volatile int abort;
  volatile int job_type, job_buf;
};

// The barriers live after the buffers in dynamic shared memory (no static shared memory, so
// the dynamic window starts 1024-byte aligned, as the swizzled tiles need, without padding).
constexpr int kSmemBytes = kSideMax + (int)((sizeof(Shared) + 15) / 16 * 16);

// A work item is a piece of a 128-row tile's key sweep: 128-key steps s0 .. s1-1.  A tile
// cut into several pieces (np > 1) has them written as partial results (the output
// normalised by the piece's own softmax sum, and its log-sum-exp) into consecutive slots
// from `base`; merge_kernel combines them after the attention kernel.
struct Item {
  int b, t, P, nb;
  int ns;   // 128-key steps: ceil(nb / 2)
  int rot;  // first step of this tile's sweep (see decode)
  int np, slot, base;
  int64_t k0, k1;
  bool bad;
};

// Work item k of the schedule, from its two 16-byte records.
__device__ __forceinline__ int4 item_rec(const TcParams& p, int item, int h) {
  return __ldg(p.items + 2 * item + h);
}

__device__ __noinline__ Item decode_info(const TcParams& p, int4 a, int4 v) {
  Item it;
  it.b = a.x;
  it.t = a.y;
  it.P = v.x;
  it.np = v.y;
  it.slot = v.z;
  it.base = v.w;
  const int64_t kv_len = (int64_t)it.P + p.Q;
  it.bad = it.P < 0 || it.P > p.max_prefix || kv_len > p.seq_cap;
  int64_t kend = kv_len;
  if (p.causal) {
    // no row of the tile sees past its last row's node
    const int64_t hi = ((int64_t)(it.t + 1) * kRows - 1) / p.H;
    kend = (int64_t)it.P + (hi < p.Q - 1 ? hi : p.Q - 1) + 1;
  }
  it.k0 = (int64_t)a.z * kStep;
  int64_t k1 = (int64_t)a.w * kStep < kend ? (int64_t)a.w * kStep : kend;
  if (it.bad || k1 < it.k0) k1 = it.k0;
  it.k1 = k1;
  it.nb = k1 > it.k0 ? (int)((k1 - it.k0 + kBN - 1) / kBN) : 0;
  it.ns = (it.nb + 1) >> 1;
  // The row tiles of one sequence run at the same time on neighbouring clusters; a whole
  // tile starts its sweep over the key steps at a step of its own so that they do not all
  // request the same cache lines at once (the softmax is independent of block order).
  it.rot = (it.ns > 0 && a.z == 0 && k1 == kend) ? (int)(((int64_t)it.t * it.ns) / p.tiles_per_seq)
                                                  : 0;
  return it;
}

__device__ __forceinline__ Item decode(const TcParams& p, int item) {
  return decode_info(p, item_rec(p, item, 0), item_rec(p, item, 1));
}

// Item taken by cluster `cid` in round r, or -1 when it has none left (each cluster works
// through its own list of the schedule, see schedule_kernel).
__device__ __forceinline__ int item_at(const TcParams& p, int r, int cid, int) {
  const int k = __ldg(p.cl_start + cid) + r;
  return k < __ldg(p.cl_start + cid + 1) ? k : -1;
}

// 128-key step visited at position j of the tile's sweep; it holds the 64-key blocks
// 2*step and (if it exists) 2*step + 1.
__device__ __forceinline__ int sweep_step(const Item& it, int j) {
  const int jj = j + it.rot;
  return jj >= it.ns ? jj - it.ns : jj;
}

// Cache row of key `key` (relative to the item's first key) of a contiguous cache.
__device__ __forceinline__ int64_t key_row(const TcParams& p, const Item& it, int64_t key) {
  return (int64_t)it.b * p.seq_rows + it.k0 + key;
}

// Cache row of the first key of 64-key block `blk` (relative to the item's first key).
__device__ __forceinline__ int64_t block_row(const TcParams& p, const Item& it, int blk) {
  if (!p.paged) return key_row(p, it, (int64_t)blk * kBN);
  const int64_t lb = (it.k0 >> 6) + blk;
  return (int64_t)__ldg(p.page_table + (int64_t)it.b * p.max_pages + lb) * kBN;
}

// Index of a step's tensor maps / swap flag (paged cache).
__device__ __forceinline__ int64_t step_index(const TcParams& p, const Item& it, int step) {
  return (int64_t)it.b * p.steps_per_seq + (it.k0 >> 7) + step;
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
    if (globaltimer() - t0 > sh.timeout_ns) {
      raise_abort(sh, status, TV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Exit drain: wait for phase `parity` of a barrier that asynchronous work (a TMA load, the
// tensor cores) still has to complete, whether or not the kernel is aborting, so that no
// copy or MMA is in flight when the CTA frees its tensor memory and leaves.  Bounded by its
// own deadline; if that runs out the kernel reports TV_ERR_TIMEOUT and leaves anyway.
__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer() - t0 > kDrainNs) {
      report(status, TV_ERR_TIMEOUT);
      return;
    }
  }
}

// Drain a ring of n stages whose full barriers got `count` loads so far: the last issue of
// each stage may still be in flight (earlier ones were consumed before it was re-armed).
__device__ __noinline__ void drain_ring(uint64_t* full, uint32_t n, uint32_t count,
                                        int32_t* status) {
  for (uint32_t k = 0; k < n && k < count; ++k) {
    const uint32_t u = count - 1 - k;
    drain_wait(&full[u % n], (u / n) & 1, status);
  }
}

__device__ __forceinline__ bool wait_bar(Shared& sh, uint64_t* bar, uint32_t parity,
                                         int32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  return wait_bar_slow(sh, a, parity, status);
}

// Same, for a barrier that only this CTA's threads, TMA loads and MMAs complete.
__device__ __forceinline__ bool wait_bar_cta(Shared& sh, uint64_t* bar, uint32_t parity,
                                             int32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cta(a, parity)) return true;
  return wait_bar_slow(sh, a, parity, status);
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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One 64-key half of a step: p = 2^(s*c - mr) for the 64 scores (masked ones are -inf),
// packed to bf16 into this row of a staging buffer (swizzled K-major layout); returns the
// sum.
__device__ __forceinline__ float emit_half(const float* t, float c, float mr, unsigned char* row,
                                           uint32_t sw) {
  const uint64_t cc = f2_pack(c, c), nm = f2_pack(-mr, -mr);
  uint64_t s2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x0, x1;
      f2_unpack(f2_fma(f2_pack(t[8 * q + 2 * e], t[8 * q + 2 * e + 1]), cc, nm), x0, x1);
      const float p0 = ex2(x0), p1 = ex2(x1);
      s2[e & 1] = f2_add(s2[e & 1], f2_pack(p0, p1));
      w[e] = pack_bf16(p0, p1);
    }
    *reinterpret_cast<uint4*>(row + (((uint32_t)q ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  float a0, a1, b0, b1;
  f2_unpack(s2[0], a0, a1);
  f2_unpack(s2[1], b0, b1);
  return (a0 + a1) + (b0 + b1);
}

// Masked keys of a 64-key half get score -inf.
__device__ __forceinline__ void apply_mask(float* t, uint64_t vis) {
  if (vis == ~0ull) return;
  const uint32_t lo = (uint32_t)vis, hi = (uint32_t)(vis >> 32);
#pragma unroll
  for (int k = 0; k < 32; ++k) t[k] = ((lo >> k) & 1u) ? t[k] : -INFINITY;
#pragma unroll
  for (int k = 0; k < 32; ++k) t[32 + k] = ((hi >> k) & 1u) ? t[32 + k] : -INFINITY;
}

// ===================================================================================
// rank 0: QK^T + softmax
// ===================================================================================
__device__ void s_side(const TcParams& p, const CUtensorMap* map_lat, const CUtensorMap* map_kpe,
                       const CUtensorMap* map_q, const CUtensorMap* map_qr, Shared& sh,
                       unsigned char* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* lat = smem;
  unsigned char* rope = smem + kRopeOff;
  unsigned char* qrope = smem + kQropeOff;
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer: four latent boxes and the rope box per step --------
    // Each tile starts with its latent queries, which pass through the key ring (the same
    // four box shapes) on their way into TMEM, and its rope queries, which go straight to
    // their buffer once the previous tile's MMAs are done with it.
    if (lane == 0) {
      prefetch_tensormap(map_lat);
      prefetch_tensormap(map_kpe);
      prefetch_tensormap(map_q);
      prefetch_tensormap(map_qr);
      // The refill latency of the rings is on the critical path: each cache layout gets its
      // own lean loop (the branch is taken once per tile).
      uint32_t u = 0, rc = 0, qi = 0;
      auto produce = [&]() {
      for (int rr = 0, item; (item = item_at(p, rr, cid, ncl)) >= 0 && !sh.abort; ++rr) {
        const Item it = decode(p, item);
        if (it.ns == 0) continue;
        const int qrow0 = it.b * p.Q * p.H + it.t * kRows;
        for (int h = 0; h < 4; ++h, ++u) {
          const uint32_t st = u % kNLS;
          if (!wait_bar(sh, &sh.slat_empty[st], ((u / kNLS) & 1) ^ 1, p.status)) return;
          mbar_arrive_expect_tx(&sh.slat_full[st], kStageS);
          tma_load_3d(lat + st * kStageS, map_q, 0, qrow0, 2 * h, &sh.slat_full[st]);
        }
        if (!wait_bar_cta(sh, &sh.q_free, (qi & 1) ^ 1, p.status)) return;
        ++qi;
        mbar_arrive_expect_tx(&sh.qr_full, kChunkS);
        tma_load_2d(qrope, map_qr, 0, qrow0, &sh.qr_full);
        if (!p.paged) {
          for (int j = 0; j < it.ns; ++j, ++rc) {
            const int row0 = (int)key_row(p, it, (int64_t)sweep_step(it, j) * kStep);
            for (int h = 0; h < 4; ++h, ++u) {
              const uint32_t st = u % kNLS;
              if (!wait_bar(sh, &sh.slat_empty[st], ((u / kNLS) & 1) ^ 1, p.status)) return;
              mbar_arrive_expect_tx(&sh.slat_full[st], kStageS);
              tma_load_3d(lat + st * kStageS, map_lat, 0, row0, 2 * h, &sh.slat_full[st]);
            }
            const uint32_t rs = rc % kNRope;
            if (!wait_bar(sh, &sh.rope_empty[rs], ((rc / kNRope) & 1) ^ 1, p.status)) return;
            mbar_arrive_expect_tx(&sh.rope_full[rs], kChunkS);
            tma_load_2d(rope + rs * kChunkS, map_kpe, 0, row0, &sh.rope_full[rs]);
          }
          continue;
        }
        // paged cache: per-step maps, written by prep_kernel; acquired for the whole tile
        // up front, each step's prefetched one step ahead
        const CUtensorMap* mb = p.step_maps + 2 * step_index(p, it, 0);
        for (int jj = 0; jj < it.ns; ++jj) {
          tmap_acquire(mb + 2 * jj);
          tmap_acquire(mb + 2 * jj + 1);
        }
        if (it.ns > 0) {
          prefetch_tensormap(mb + 2 * sweep_step(it, 0));
          prefetch_tensormap(mb + 2 * sweep_step(it, 0) + 1);
        }
        for (int j = 0; j < it.ns; ++j, ++rc) {
          const CUtensorMap* ml = mb + 2 * sweep_step(it, j);
          if (j + 1 < it.ns) {
            const CUtensorMap* mn = mb + 2 * sweep_step(it, j + 1);
            prefetch_tensormap(mn);
            prefetch_tensormap(mn + 1);
          }
#pragma unroll 1
          for (int h = 0; h < 4; ++h, ++u) {
            const uint32_t st = u % kNLS;
            if (!wait_bar(sh, &sh.slat_empty[st], ((u / kNLS) & 1) ^ 1, p.status)) return;
            mbar_arrive_expect_tx(&sh.slat_full[st], kStageS);
            tma_load_5d(lat + st * kStageS, ml, 0, 0, 0, 0, 2 * h, &sh.slat_full[st]);
          }
          const uint32_t rs = rc % kNRope;
          if (!wait_bar(sh, &sh.rope_empty[rs], ((rc / kNRope) & 1) ^ 1, p.status)) return;
          mbar_arrive_expect_tx(&sh.rope_full[rs], kChunkS);
          tma_load_4d(rope + rs * kChunkS, ml + 1, 0, 0, 0, 0, &sh.rope_full[rs]);
        }
      }
      };
      if (!p.test_skip_loads) produce();
      // leave no load in flight (after an abort the consumers stop taking stages; in a
      // normal run these phases have completed already)
      drain_ring(sh.slat_full, kNLS, u, p.status);
      drain_ring(sh.rope_full, kNRope, rc, p.status);
      drain_ring(&sh.qr_full, 1, qi, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: S = Q K^T, 128 keys per step ----------------------
    if (lane == 0) {
      // The issuing thread must keep the tensor pipe's queue fed, so its loop is kept lean:
      // stage index, phase and descriptor advance incrementally, and the MMAs of a stage
      // add constant offsets to one descriptor (address bits 4..17 sit in its low field,
      // which these offsets never overflow).
      uint32_t sc = 0, qc = 0, rc = 0, st = 0, sph = 0;
      const uint64_t dq = smem_desc(smem_u32(qrope), 16, 1024, 2);
      const uint64_t dr = smem_desc(smem_u32(rope), 16, 1024, 2);
      const uint64_t dl0 = smem_desc(smem_u32(lat), 16, 1024, 2);
      uint64_t db = dl0;
      for (int rr = 0, item; (item = item_at(p, rr, cid, ncl)) >= 0 && !sh.abort; ++rr) {
        const Item it = decode(p, item);
        if (it.ns == 0) continue;
        // The tile's latent queries arrive through the key ring as four stages; they are
        // copied into TMEM once the previous tile's MMAs have finished reading it.
        if (!wait_bar_cta(sh, &sh.q_free, (qc & 1) ^ 1, p.status)) break;
        tc_fence_after();
        bool okq = true;
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          if (!wait_bar_cta(sh, &sh.slat_full[st], sph, p.status)) { okq = false; break; }
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tmem_cp_128x256b(tmem + kTmQ + 32 * (2 * h + c) + 8 * kk,
                               db + (uint64_t)((c * kChunkS + 32 * kk) >> 4));
          mma_commit(&sh.slat_empty[st]);
          db += kStageS >> 4;
          if (++st == kNLS) {
            st = 0;
            sph ^= 1;
            db = dl0;
          }
        }
        if (!okq || !wait_bar_cta(sh, &sh.qr_full, qc & 1, p.status)) break;
        // (no abort test in the loop condition: every wait below returns false once the
        // abort flag is up, and a shared-memory load per step on this thread's critical
        // path cost about 3 % of the whole kernel)
        for (int j = 0; j < it.ns; ++j, ++sc, ++rc) {
          const uint32_t sb = sc & 1;
          if (!wait_bar_cta(sh, &sh.s_empty[sb], ((sc >> 1) & 1) ^ 1, p.status)) break;
          tc_fence_after();  // the softmax warps' TMEM reads of this S buffer come first
          const uint32_t d = tmem + (sb ? kTmS1 : kTmS0);
          bool ok = true;
          // (one stage per iteration, not unrolled: see the note on code size in the softmax)
#pragma unroll 1
          for (int h = 0; h < 4; ++h) {
            if (!wait_bar_cta(sh, &sh.slat_full[st], sph, p.status)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(d, tmem + kTmQ + 32 * (2 * h + c) + 8 * kk,
                       db + (uint64_t)((c * kChunkS + 32 * kk) >> 4), kIdescQK, (h | c | kk) != 0);
            mma_commit(&sh.slat_empty[st]);
            db += kStageS >> 4;
            if (++st == kNLS) {
              st = 0;
              sph ^= 1;
              db = dl0;
            }
          }
          static_assert(kNRope == 1, "one rope stage");
          if (!ok || !wait_bar_cta(sh, &sh.rope_full[0], rc & 1, p.status)) break;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, dq + (uint64_t)((32 * kk) >> 4), dr + (uint64_t)((32 * kk) >> 4), kIdescQK, 1);
          mma_commit(&sh.rope_empty[0]);
          mma_commit(&sh.s_full[sb]);
        }
        mma_commit(&sh.q_free);
        ++qc;
      }
      // every MMA and TMEM copy this thread issued completes before tensor memory is freed
      mma_commit(&sh.final_bar);
      drain_wait(&sh.final_bar, 0, p.status);
    }
  } else if (warp >= 4) {
    // ---------------- softmax warpgroup: thread r owns tile row r ------------------
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float c = p.scale_log2;
    const uint32_t peer = cluster_rank() ^ 1u;
    // the peer's inbox; this row's place in a message (swizzled K-major P)
    const uint32_t inbox_peer = map_to_rank(smem_u32(smem + kInboxOff), peer);
    unsigned char* stg = smem + kStgOff;
    const uint32_t row_off = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
    const uint32_t sw = (uint32_t)(r & 7);
    bool ok0 = true;  // thread 0: its last inbox waits and copies went through
    // The four warps leave their loops only together, at a 128-thread barrier that agrees
    // on the outcome of the waits before it (a warp that left alone would strand the
    // others at the next barrier).
    uint32_t sc = 0, mc = 0;
    bool live = true;
    // The next item's record is requested a whole tile ahead (its queries reach TMEM
    // without these warps).
    int item_next = item_at(p, 0, cid, ncl);
    int4 info_next = item_next >= 0 ? item_rec(p, item_next, 0) : make_int4(0, 0, 0, 0);
    int4 info_next2 = item_next >= 0 ? item_rec(p, item_next, 1) : make_int4(0, 0, 0, 0);
    for (int rr = 0; item_next >= 0 && live; ++rr) {
      const Item it = decode_info(p, info_next, info_next2);
      item_next = item_at(p, rr + 1, cid, ncl);
      if (item_next >= 0) {
        info_next = item_rec(p, item_next, 0);
        info_next2 = item_rec(p, item_next, 1);
      }
      const int trow = it.t * kRows + r;
      const bool vrow = trow < p.Q * p.H;
      const int64_t grow = (int64_t)it.b * p.Q * p.H + trow;
      // a whole tile's lse goes to the output; a piece's to its slot
      float* lse_dst = it.np == 1 ? p.lse + grow : p.ws_lse + (int64_t)it.slot * kRows + r;
      if (it.nb == 0) continue;  // nothing to compute: the O side writes the empty result
      const int node = trow / p.H;
      const uint64_t anc = (vrow && !p.causal) ? p.anc[(int64_t)it.b * p.Q + node] : 0ull;
      // every key below pv is visible: the prefix, or for a causal row all keys up to its own
      const int64_t pv = p.causal ? (int64_t)it.P + node + 1 : (int64_t)it.P;
      const int64_t k1 = it.k1;


      float m = -INFINITY, l = 0.f;
      uint32_t swap_next =
          (p.paged && __ldg(p.step_swap + step_index(p, it, sweep_step(it, 0)))) ? 64u : 0u;
      for (int j = 0; j < it.ns; ++j, ++sc) {
        if (j == (it.ns > 3 ? it.ns - 3 : 0) && item_next >= 0) {
          // warm L2 with the next tile's queries a few steps before they are needed (the
          // key stream would evict lines fetched much earlier)
          const int nrow = info_next.y * kRows + r;
          if (nrow < p.Q * p.H) {
            const int64_t ng = (int64_t)info_next.x * p.Q * p.H + nrow;
            const char* qlp = reinterpret_cast<const char*>(p.q_latent + ng * kDL);
#pragma unroll
            for (int l128 = 0; l128 < 8; ++l128) prefetch_l2(qlp + 128 * l128);
            prefetch_l2(p.q_pe + ng * kDR);
          }
        }
        const uint32_t sb = sc & 1;
        // each warp agrees before its warp-collective TMEM loads
        const bool okf =
            __all_sync(0xffffffffu, wait_bar(sh, &sh.s_full[sb], (sc >> 1) & 1, p.status));
        float t[128];
        const int st = sweep_step(it, j);
        // paged cache: a step whose second page lies below its first holds the second
        // page's keys in S columns 0..63 (the flag is read a step ahead)
        const uint32_t sw64 = swap_next;
        if (p.paged && j + 1 < it.ns)
          swap_next = __ldg(p.step_swap + step_index(p, it, sweep_step(it, j + 1))) ? 64u : 0u;
        if (!okf) {
#pragma unroll
          for (int k = 0; k < 128; ++k) t[k] = 0.f;
        } else {
          tc_fence_after();
          uint32_t sr[128];
          const uint32_t ta = tmem + lane_base + (sb ? kTmS1 : kTmS0);
          tmem_ld32(ta + sw64, sr);
          tmem_ld32(ta + sw64 + 32, sr + 32);
          tmem_ld32(ta + (sw64 ^ 64u), sr + 64);
          tmem_ld32(ta + (sw64 ^ 64u) + 32, sr + 96);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 128; ++k) t[k] = __uint_as_float(sr[k]);
        }
        const bool two = 2 * st + 1 < it.nb;
        const int64_t key0 = it.k0 + (int64_t)st * kStep;
        const uint64_t vis0 =
            (key0 + kBN > pv || key0 + kBN > k1) ? block_vis(key0, pv, k1, anc) : ~0ull;
        const uint64_t vis1 =
            !two ? 0ull
                 : ((key0 + 2 * kBN > pv || key0 + 2 * kBN > k1)
                        ? block_vis(key0 + kBN, pv, k1, anc)
                        : ~0ull);
        apply_mask(t, vis0);
        apply_mask(t + 64, vis1);
        float mx;
        {
          // 128 -> 43 -> 15 -> 5 -> 2 -> 1 with three-input maxima
          float a[43];
#pragma unroll
          for (int i = 0; i < 42; ++i) a[i] = fmax3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
          a[42] = fmaxf(t[126], t[127]);
#pragma unroll
          for (int i = 0; i < 14; ++i) a[i] = fmax3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
          a[14] = a[42];
#pragma unroll
          for (int i = 0; i < 5; ++i) a[i] = fmax3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
          mx = fmax3(a[0], a[1], fmaxf(a[2], fmaxf(a[3], a[4]))) * c;  // block max in log2 units
        }
        // The running max m moves only when the block max exceeds it by more than 2^8;
        // then O and l are rescaled by alpha = 2^(m_old - m_new).
        float alpha = 1.f;
        if (mx > (m == -INFINITY ? -INFINITY : m + kRescaleThreshold)) {
          if (l > 0.f) alpha = ex2(m - mx);
          m = mx;
        }
        const float mr = m == -INFINITY ? 0.f : m;

        // ---- messages: P, alpha, l into the two staging buffers, then bulk copies ----
        // Thread 0 issued the previous step's copies; once they have read the staging
        // buffers, the barrier below lets everyone overwrite them.  The barriers also OR
        // the rescale flag and agree on whether to go on.
        if (r == 0) bulk_wait_read<0>();
        const bool resc = named_sync_or(1, 128, alpha != 1.f);
        if (!named_sync_and(2, 128, okf && ok0 && !sh.abort)) {
          live = false;
          break;
        }
        unsigned char* stg1 = stg + kMsgBytes;
        // Code size matters here: the S side's hot loops (producer, MMA issue, softmax) run
        // on one SM at once, and when they outgrow its instruction cache the misses of all
        // its SMs queue at the GPC's shared cache (measured: 80 % of that cache's request
        // rate, 25 % of fetches missing, every SM pair slowed by where it sits in the GPC).
        // So the two 64-key halves go through one copy of the exponent code, each half's
        // scores read from tensor memory again (the registers above are only for the max);
        // the S buffer is released after that second read.
        float sum = 0.f;
        {
          const uint32_t ta = tmem + lane_base + (sb ? kTmS1 : kTmS0);
#pragma unroll 1
          for (int hh = 0; hh < (two ? 2 : 1); ++hh) {
            uint32_t hr[64];
            float h64[64];
            const uint32_t col = hh ? (sw64 ^ 64u) : sw64;
            tmem_ld32(ta + col, hr);
            tmem_ld32(ta + col + 32, hr + 32);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 64; ++k) h64[k] = __uint_as_float(hr[k]);
            apply_mask(h64, hh ? vis1 : vis0);
            sum += emit_half(h64, c, mr, stg + hh * kMsgBytes + row_off, sw);
          }
          tc_fence_before();
          mbar_arrive(&sh.s_empty[sb]);
        }
        l = l * alpha + sum;
        reinterpret_cast<float*>(stg + kMsgAlpha)[r] = alpha;
        reinterpret_cast<float*>(stg + kMsgL)[r] = l;
        if (r == 0) *reinterpret_cast<uint4*>(stg + kMsgFlags) = make_uint4(resc ? kFlagRescale : 0u, 0u, 0u, 0u);
        if (two) {
          reinterpret_cast<float*>(stg1 + kMsgAlpha)[r] = 1.f;
          reinterpret_cast<float*>(stg1 + kMsgL)[r] = l;
          if (r == 0) *reinterpret_cast<uint4*>(stg1 + kMsgFlags) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (j == it.ns - 1 && vrow)  // the tile's (or piece's) log-sum-exp
          *lse_dst = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        fence_proxy_async_smem();  // the bulk copies read the staging through the async proxy
        named_sync(3, 128);
        if (r == 0) {
          // each message goes to the next inbox buffer once rank 1 has released it
          for (int k = 0; k < (two ? 2 : 1) && ok0; ++k) {
            const uint32_t mk = mc + k, ib = mk % kNInbox;
            ok0 = wait_bar(sh, &sh.pdst_free[ib], ((mk / kNInbox) & 1) ^ 1, p.status);
            if (ok0)
              bulk_copy_to_cluster(inbox_peer + ib * kMsgStride, stg + k * kMsgBytes, kMsgBytes,
                                   map_to_rank(smem_u32(&sh.p_full[ib]), peer));
          }
          bulk_commit();
        }
        mc += two ? 2 : 1;
      }
      if (!live) break;
    }
    if (r == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
}

// ===================================================================================
// rank 1: O += P V, rescale, epilogue
// ===================================================================================
__device__ void o_side(const TcParams& p, const CUtensorMap* map_lat, Shared& sh,
                       unsigned char* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* lat = smem;
  unsigned char* inbox = smem + kInboxOff;
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer: each 64-key block's latent chunks, in message order --
    if (lane == 0) {
      prefetch_tensormap(map_lat);
      uint32_t u = 0;
      auto produce = [&]() {
      for (int rr = 0, item; (item = item_at(p, rr, cid, ncl)) >= 0 && !sh.abort; ++rr) {
        const Item it = decode(p, item);
        // cache rows of each step's blocks are looked up a step ahead
        int rows_next[2] = {0, 0};
        if (it.ns > 0) {
          const int s0 = sweep_step(it, 0);
          rows_next[0] = (int)block_row(p, it, 2 * s0);
          if (2 * s0 + 1 < it.nb) rows_next[1] = (int)block_row(p, it, 2 * s0 + 1);
        }
        for (int j = 0; j < it.ns; ++j) {
          const int st = sweep_step(it, j);
          const int nh = 2 * st + 1 < it.nb ? 2 : 1;
          const int rows_cur[2] = {rows_next[0], rows_next[1]};
          if (j + 1 < it.ns) {
            const int s1 = sweep_step(it, j + 1);
            rows_next[0] = (int)block_row(p, it, 2 * s1);
            if (2 * s1 + 1 < it.nb) rows_next[1] = (int)block_row(p, it, 2 * s1 + 1);
          }
          for (int hh = 0; hh < nh; ++hh) {
            const int row0 = rows_cur[hh];
            for (int h = 0; h < 2; ++h, ++u) {
              const uint32_t ls = u % kNLO;
              if (!wait_bar(sh, &sh.olat_empty[ls], ((u / kNLO) & 1) ^ 1, p.status)) return;
              mbar_arrive_expect_tx(&sh.olat_full[ls], kHalfO);
              tma_load_3d(lat + ls * kHalfO, map_lat, 0, row0, 4 * h, &sh.olat_full[ls]);
            }
          }
        }
      }
      };
      produce();
      drain_ring(sh.olat_full, kNLO, u, p.status);  // no load left in flight
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: O += P V ------------------------------------------
    if (lane == 0) {
      const uint32_t peer = cluster_rank() ^ 1u;
      uint32_t vc = 0, mc = 0, ic = 0, dc = 0, cc = 0, last_pb = 0;
      for (int rr = 0, item; (item = item_at(p, rr, cid, ncl)) >= 0 && !sh.abort; ++rr) {
        const Item it = decode(p, item);
        if (it.nb == 0) continue;
        if (ic > 0) {
          // the previous tile's epilogue has read its last message: hand that buffer back
          if (!wait_bar(sh, &sh.epi_done, (ic - 1) & 1, p.status)) break;
          mbar_arrive_remote(map_to_rank(smem_u32(&sh.pdst_free[last_pb]), peer));
        }
        tc_fence_after();
        bool ok = true;
        for (int j = 0; j < it.nb && ok; ++j, ++mc) {
          const uint32_t pb = mc % kNInbox;
          last_pb = pb;
          if (!wait_bar(sh, &sh.p_full[pb], (mc / kNInbox) & 1, p.status)) { ok = false; break; }
          // arm the buffer's next phase now: its next message is only sent after the MMAs
          // below have read this one
          mbar_arrive_expect_tx(&sh.p_full[pb], kMsgBytes);
          // The message arrived by a bulk copy, in the async proxy the MMAs read through, so
          // this fence is not required for ordering; a variant without it (flags loaded
          // before the re-arm) measured about 1 % slower, so it stays.
          fence_proxy_async_smem();
          const uint32_t flags =
              *reinterpret_cast<volatile uint32_t*>(inbox + pb * kMsgStride + kMsgFlags);
          if (j > 0 && (flags & kFlagRescale)) {
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
            const uint32_t va = smem_u32(lat + st * kHalfO);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + 256 * h, smem_desc(pa + 32 * kk, 16, 1024, 2),
                     smem_desc(va + 2048 * kk, 8192, 1024, 2), kIdescPV, (j | kk) != 0);
            mma_commit(&sh.olat_empty[st]);
          }
          // once the MMAs have read the message, the buffer goes straight back to rank 0's
          // softmax; a tile's last message stays until the epilogue has read its row sums
          if (j < it.nb - 1) mma_commit_multicast(&sh.pdst_free[pb], (uint16_t)(1u << peer));
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
      drain_wait(&sh.final_bar, 0, p.status);
    }
  } else if (warp >= 4) {
    // ---------------- rescale / epilogue warpgroup: thread r owns tile row r -------
    const int wq = warp - 4;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    uint32_t jc = 0;
    for (int rr = 0, item; (item = item_at(p, rr, cid, ncl)) >= 0 && !sh.abort; ++rr) {
      const Item it = decode(p, item);
      const int trow = it.t * kRows + r;
      const bool vrow = trow < p.Q * p.H;
      const int64_t grow = (int64_t)it.b * p.Q * p.H + trow;
      // a whole tile goes to the output, a piece of a split tile to its slot
      float* dst = it.np == 1 ? p.out + grow * kDL
                              : p.ws_out + ((int64_t)it.slot * kRows + r) * kDL;
      if (it.bad && r == 0) report(p.status, TV_ERR_BOUNDS);
      if (it.nb == 0) {
        // no visible key in this item (an empty piece or an out-of-range prefix)
        if (vrow) {
          for (int c = 0; c < kDL / 4; ++c)
            reinterpret_cast<float4*>(dst)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          *(it.np == 1 ? p.lse + grow : p.ws_lse + (int64_t)it.slot * kRows + r) = -INFINITY;
        }
      }
      for (; it.nb > 0;) {
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
          // Each thread holds its own row (TMEM lane), so storing straight from registers
          // would make every warp store touch 32 rows.  Each 32-row x 32-column chunk is
          // staged in shared memory instead (16-byte pieces XOR-swizzled by row, so that both
          // the writes and the reads below are free of bank conflicts) and written back with
          // lanes along the columns: every store instruction fills four whole 128-byte lines.
          float* stg = reinterpret_cast<float*>(smem + kEpiOff) + wq * 1024;
          const int wrow0 = it.t * kRows + wq * 32;  // tile row of this warp's lane 0
          const int rows_ok = p.Q * p.H - wrow0;     // valid rows of the warp's 32
          float* dst0 = dst - (int64_t)lane * kDL;   // row of lane 0
          const int rr4 = lane >> 3, jj = lane & 7;
          auto put_chunk = [&](const uint32_t* v, int c) {
            __syncwarp();  // the previous chunk's reads of the staging are done
#pragma unroll
            for (int e = 0; e < 8; ++e)
              *reinterpret_cast<float4*>(stg + lane * 32 + ((e ^ (lane & 7)) << 2)) =
                  make_float4(__uint_as_float(v[4 * e]) * inv, __uint_as_float(v[4 * e + 1]) * inv,
                              __uint_as_float(v[4 * e + 2]) * inv, __uint_as_float(v[4 * e + 3]) * inv);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int row = 4 * i + rr4;
              const float4 x = *reinterpret_cast<const float4*>(stg + row * 32 + ((jj ^ (row & 7)) << 2));
              if (row < rows_ok)
                *reinterpret_cast<float4*>(dst0 + (int64_t)row * kDL + 32 * c + 4 * jj) = x;
            }
          };
          // two chunks in flight: each TMEM load overlaps the previous chunk's stores
          uint32_t va[32], vb[32];
          tmem_ld32(tmem + lane_base, va);
          tmem_wait_ld_regs(va);
#pragma unroll 1
          for (int c = 0; c < 16; c += 2) {
            tmem_ld32(tmem + lane_base + 32 * (c + 1), vb);
            put_chunk(va, c);
            tmem_wait_ld_regs(vb);
            if (c + 2 < 16) tmem_ld32(tmem + lane_base + 32 * (c + 2), va);
            put_chunk(vb, c + 1);
            if (c + 2 < 16) tmem_wait_ld_regs(va);
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
attn_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap map_lat_s,
               const __grid_constant__ CUtensorMap map_kpe_s,
               const __grid_constant__ CUtensorMap map_lat_o,
               const __grid_constant__ CUtensorMap map_q,
               const __grid_constant__ CUtensorMap map_qr) {
  extern __shared__ __align__(1024) unsigned char smem[];
  if (smem_u32(smem) & 1023u) {  // both CTAs see the same layout, so both leave here
    if (threadIdx.x == 0) report(p.status, TV_ERR_UNSUPPORTED);
    return;
  }
  Shared& sh = *reinterpret_cast<Shared*>(smem + kSideMax);
  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNLS; ++i) {
      mbar_init(&sh.slat_full[i], 1);
      mbar_init(&sh.slat_empty[i], 1);
    }
    for (int i = 0; i < kNLO; ++i) {
      mbar_init(&sh.olat_full[i], 1);
      mbar_init(&sh.olat_empty[i], 1);
    }
    for (int i = 0; i < kNRope; ++i) {
      mbar_init(&sh.rope_full[i], 1);
      mbar_init(&sh.rope_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.s_empty[i], 128);
    }
    for (int i = 0; i < kNInbox; ++i) {
      mbar_init(&sh.pdst_free[i], 1);
      mbar_init(&sh.p_full[i], 1);
    }
    mbar_init(&sh.qr_full, 1);
    mbar_init(&sh.q_free, 1);
    mbar_init(&sh.drain, 1);
    mbar_init(&sh.job_full, 1);
    mbar_init(&sh.corr_done, 128);
    mbar_init(&sh.epi_done, 128);
    mbar_init(&sh.final_bar, 1);
    sh.abort = 0;
    sh.timeout_ns = p.timeout_ns;
    sh.job_type = 0;
    sh.job_buf = 0;
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
  cluster_sync();  // barriers of both CTAs exist before any remote arrive or store
  // The kernel may start while prep_kernel (just before it in the stream) still runs
  // (programmatic dependent launch): the set-up above overlaps it, and everything below
  // reads its work records and step maps only after this wait.
  griddep_wait();

  if (rank == 0)
    s_side(p, &map_lat_s, &map_kpe_s, &map_q, &map_qr, sh, smem);
  else
    o_side(p, &map_lat_o, sh, smem);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(sh.tmem_base, 512);
  if (p.test_exit_counts && threadIdx.x == 0) {
    atomicAdd(p.test_exit_counts, 1);
    if (sh.abort) atomicAdd(p.test_exit_counts + 1, 1);
  }
  cluster_sync();  // neither CTA leaves while the other may still touch its memory
}

// Copies every in-range 64-key page of a paged cache into a contiguous key view: row
// b * seq_rows + key holds c_kv (512 bf16) then k_pe (64 bf16) of that key.  One CTA per
// (page slot, sequence).  A page index that points outside the cache rows is reported as
// TV_ERR_BOUNDS and its rows are left unwritten (the sequence's result is then undefined,
// as for any out-of-range input).
__global__ void __launch_bounds__(256)
gather_kv_kernel(const uint4* __restrict__ ckv, int64_t ckv_stride16, const uint4* __restrict__ kpe,
                 int64_t kpe_stride16, const int32_t* __restrict__ page_table, int max_pages,
                 const int32_t* __restrict__ prefix_len, int Q, int max_prefix, int64_t num_rows,
                 int64_t seq_rows, uint4* __restrict__ out, int32_t* status) {
  constexpr int kW = (kDL + kDR) * 2 / 16;  // 72 16-byte words per key row
  griddep_launch_dependents();  // the attention kernel may start its prologue now
  const int b = blockIdx.y, j = blockIdx.x;
  const int P = prefix_len[b];
  if (P < 0 || P > max_prefix) return;  // reported by the attention kernel
  const int64_t kv_len = (int64_t)P + Q;
  if ((int64_t)j * kBN >= kv_len || j >= max_pages) return;
  const int64_t pg = page_table[(int64_t)b * max_pages + j];
  if (pg < 0 || (pg + 1) * kBN > num_rows) {
    if (threadIdx.x == 0) report(status, TV_ERR_BOUNDS);
    return;
  }
  const int64_t src0 = pg * kBN, dst0 = (int64_t)b * seq_rows + (int64_t)j * kBN;
#pragma unroll 2
  for (int idx = threadIdx.x; idx < kBN * kW; idx += 256) {
    const int i = idx / kW, w = idx - i * kW;
    const uint4 v = w < 64 ? __ldg(ckv + (src0 + i) * ckv_stride16 + w)
                           : __ldg(kpe + (src0 + i) * kpe_stride16 + (w - 64));
    out[(dst0 + i) * kW + w] = v;
  }
}

// ---- work schedule ---------------------------------------------------------------------
// The work is B * tiles_per_seq row tiles of 128 rows, tile (b, t) sweeping ns(b, t)
// 128-key steps.  Tiles are listed longest first: with the tree mask all tiles of a
// sequence are equally long and sequences are ranked by their key count (then tiles
// follow sequence by sequence, so that the tiles of one sequence run side by side and share
// its keys through L2); with the causal mask a tile's keys end at its last row, so tiles go
// from the last tile index down, sequences ranked within each.
//   - Automatic: the first R = floor(tiles / clusters) rounds deal whole tiles, one per
//     cluster per round, in list order, alternating direction.  With the tree mask and at
//     most kMaxRanked sequences (a list sorted longest first) the last kDealtRounds rounds
//     instead deal their tiles to the clusters in increasing order of the key steps they
//     already hold (ties by cluster index: the longest-processing-time rule, round by round
//     so that the tiles of one round still run side by side; the last three rounds dealt
//     this way even the loads about as well as all of them).  With the causal mask a
//     round's tiles differ by a step at most.  The fewer than `clusters` tiles left over
//     are cut into pieces of about equal length, at most one piece per cluster: the piece
//     length T is the smallest for which they fit, at least kMinPiece steps, and no tile is
//     cut into more than kMaxPieces pieces.  The pieces, in tile order, go to the clusters
//     that hold the fewest steps (dealt lists) or to the clusters in index order.
//   - Forced (num_splits = S): every tile in S pieces of equal step counts, the items in
//     tile order dealt to the clusters in equal contiguous runs.
// Each cluster's items are stored consecutively (cl_start[c] .. cl_start[c+1]-1;
// cl_start[ncl+1] holds the number of partial-result slots used).  The pieces of a split
// tile get consecutive slots; slot_info[slot] = {b, t, pieces, first slot}.
constexpr int kMinPiece = 4;
constexpr int kMaxPieces = 8;
constexpr int kMaxRanked = 1024;
constexpr int kMaxSchedClusters = 256;
constexpr int kDealtRounds = 3;  // whole-tile rounds dealt by load (the last ones)
constexpr int kMaxForcedSplits = 32;
// prep_kernel: threads per block (all of them compute the schedule in block 0), threads
// that write tensor maps in the other blocks, and the shared buffer (block 0: the
// schedule's lists; the other blocks: two tensor-map copies per map-writing thread)
constexpr int kPrepThreads = 1024;
constexpr int kMapThreads = 128;
constexpr int kPrepSmem = kMapThreads * 2 * 128;
static_assert(4 * kMaxRanked * 4 + 8 * kMaxSchedClusters * 4 + kDealtRounds * kMaxSchedClusters <=
                  kPrepSmem,
              "the schedule's lists must fit the prep kernel's shared buffer");
static_assert(kMaxSchedClusters <= 256, "a dealt tile's cluster is kept in one byte");
constexpr int kDealLanes = 4;  // lanes that rank one cluster in a dealt round
static_assert(kMaxSchedClusters * kDealLanes <= kPrepThreads,
              "the dealt rounds give every cluster its lanes");

struct SchedArgs {
  const int32_t* prefix_len;
  int B, Q, H, T, causal, max_prefix;
  int64_t seq_cap;
  int ncl, splits, max_slots;
  int4* items;
  int32_t* cl_start;
  int4* slot_info;
  int4* split_info;  // the merge's work list: per split tile {b, t, pieces, first slot}
  int32_t* status;
};

// 128-key steps tile t of a sequence with prefix P sweeps (0 for an out-of-range prefix)
__device__ __forceinline__ int tile_steps(const SchedArgs& a, int P, int t) {
  const int64_t kv = (int64_t)P + a.Q;
  if (P < 0 || P > a.max_prefix || kv > a.seq_cap) return 0;
  int64_t kend = kv;
  if (a.causal) {
    const int64_t hi = ((int64_t)(t + 1) * kRows - 1) / a.H;
    kend = (int64_t)P + (hi < a.Q - 1 ? hi : a.Q - 1) + 1;
  }
  return (int)((kend + kStep - 1) / kStep);
}

__device__ void schedule(const SchedArgs& a, unsigned char* buf) {
  // All scratch stays in shared memory (`buf`): fewer tiles are left over than there are
  // clusters (<= kMaxSchedClusters), and a dealt whole tile's cluster takes one byte.
  int* order = reinterpret_cast<int*>(buf);
  int* sp = order + kMaxRanked;  // prefix length of every sequence (when B <= kMaxRanked)
  int* sc = sp + kMaxRanked;     // its key steps
  int* su = sc + kMaxRanked;
  int* sbase = su + kMaxSchedClusters;
  int* rs = sbase + kMaxSchedClusters;
  int* rk = rs + kMaxSchedClusters;
  int* load = rk + kMaxSchedClusters;    // key steps a cluster holds
  int* by_rank = load + kMaxSchedClusters;  // clusters in increasing order of load
  int* rank_of = by_rank + kMaxSchedClusters;
  int* off = rank_of + kMaxSchedClusters;  // pieces on the clusters before this one
  int* ss = off + kMaxSchedClusters;       // key steps of the q-th longest sequence
  unsigned char* tcl = reinterpret_cast<unsigned char*>(ss + kMaxRanked);
  const int B = a.B, T = a.T, ncl = a.ncl;
  const int n_tiles = B * T;
  const bool ranked = B <= kMaxRanked;
  for (int i = threadIdx.x; ranked && i < B; i += blockDim.x) {
    sp[i] = a.prefix_len[i];
    sc[i] = tile_steps(a, sp[i], T - 1);
  }
  __syncthreads();
  auto P_of = [&](int b) { return ranked ? sp[b] : a.prefix_len[b]; };
  // sequences longest first (ties by index); beyond kMaxRanked the identity
  for (int i = threadIdx.x; ranked && i < B; i += blockDim.x) {
    const int ci = sc[i];
    int rank = 0;
#pragma unroll 4
    for (int j = 0; j < B; ++j) {
      const int cj = sc[j];
      rank += (cj > ci) | ((cj == ci) & (j < i));
    }
    order[rank] = i;
    ss[rank] = ci;
  }
  for (int c = threadIdx.x; c < a.ncl; c += blockDim.x) {
    load[c] = 0;
    by_rank[c] = c;
    rank_of[c] = c;
  }
  __syncthreads();
  auto seq_of = [&](int q) { return ranked ? order[q] : q; };
  // position in the longest-first tile list -> (sequence, tile)
  auto tile_at = [&](int pos, int& b, int& t) {
    if (a.causal) {
      t = T - 1 - pos / B;
      b = seq_of(pos % B);
    } else {
      t = pos % T;
      b = seq_of(pos / T);
    }
  };
  auto put = [&](int k, int b, int t, int s0, int s1, int np, int slot, int base) {
    a.items[2 * k] = make_int4(b, t, s0, s1);
    a.items[2 * k + 1] = make_int4(P_of(b), np, slot, base);
    if (slot >= 0) a.slot_info[slot] = make_int4(b, t, np, base);
  };

  if (a.splits > 0) {
    const int S = a.splits;
    const int n_items = n_tiles * S;
    for (int k = threadIdx.x; k < n_items; k += blockDim.x) {
      const int pos = k / S, j = k - pos * S;
      int b, t;
      tile_at(pos, b, t);
      const int ns = tile_steps(a, P_of(b), t);
      put(k, b, t, (int)((int64_t)j * ns / S), (int)((int64_t)(j + 1) * ns / S), S,
          S > 1 ? k : -1, S > 1 ? pos * S : -1);
      if (S > 1 && j == 0) a.split_info[pos] = make_int4(b, t, S, pos * S);
    }
    for (int c = threadIdx.x; c <= ncl; c += blockDim.x)
      a.cl_start[c] = (int)(((int64_t)c * n_items + ncl - 1) / ncl);
    if (threadIdx.x == 0) {
      a.cl_start[ncl + 1] = S > 1 ? n_items : 0;
      a.cl_start[ncl + 2] = S > 1 ? n_tiles : 0;
    }
    return;
  }

  const int R = n_tiles / ncl;  // rounds of whole tiles
  const int nd = R * ncl;
  const int nr = n_tiles - nd;  // tiles left over (fewer than ncl)
  // The last kDealtRounds rounds are dealt by load when the list is sorted longest first
  // (tree mask, ranked sequences); with the causal mask a round's tiles differ by a step at
  // most and alternating rounds do as well.
  const bool dealt = !a.causal && ranked;
  const int r0 = dealt ? max(0, R - kDealtRounds) : R;  // first dealt round
  // The dealing (threads [0, n_deal)) and the cutting of the leftover tiles (threads
  // [pb, blockDim)) share nothing: they run side by side when enough warps are left over
  // for the second, else one after the other.
  const int n_deal = dealt ? (ncl * kDealLanes + 31) / 32 * 32 : 0;
  const int pb = dealt && n_deal + 128 <= (int)blockDim.x ? n_deal : 0;
  if (dealt) {
    // kDealLanes lanes own each cluster (cluster q: threads kDealLanes*q and on) and keep its
    // load and rank in registers; the loads are shared through two arrays in turn, one read
    // while the other is written, and the warps that own clusters meet at a named barrier
    // once a dealt round.  With the tree mask every tile of a sequence sweeps the same
    // steps: list position pos sweeps ss[pos / T].  The ranking, by (load, index), is
    // redone only when the order may have changed since it was last taken (a round of equal
    // tiles adds the same to every load; in the sorted list equal first and last tiles make
    // such a round).
    const int q = (int)threadIdx.x / kDealLanes, sub = (int)threadIdx.x % kDealLanes;
    if ((int)threadIdx.x < n_deal) {
      // the key steps of the alternating rounds before r0, summed over the owner's lanes
      int my_load = 0;
      if (q < ncl)
        for (int r = sub; r < r0; r += kDealLanes)
          my_load += ss[(r * ncl + ((r & 1) ? ncl - 1 - q : q)) / T];
#pragma unroll
      for (int o = kDealLanes / 2; o > 0; o >>= 1)
        my_load += __shfl_xor_sync(0xffffffffu, my_load, o);
      int my_rank = q;
      int* cur = load;
      int* nxt = off;  // off is computed later
      if (q < ncl && sub == 0) cur[q] = my_load;
      named_sync(1, (uint32_t)n_deal);
      auto rank_own = [&]() {
        int n = 0;
        if (q < ncl) {
#pragma unroll 4
          for (int j = sub; j < ncl; j += kDealLanes) {
            const int lj = cur[j];
            n += (lj < my_load) | ((lj == my_load) & (j < q));
          }
        }
#pragma unroll
        for (int o = kDealLanes / 2; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
        my_rank = n;
      };
      bool stale = r0 > 0;
      for (int r = r0; r < R; ++r) {
        const int first = ss[(r * ncl) / T];
        const int last = ss[(r * ncl + ncl - 1) / T];
        if (stale) rank_own();
        if (q < ncl) {
          const int pos = r * ncl + my_rank;
          my_load += ss[pos / T];
          if (sub == 0) {
            nxt[q] = my_load;
            tcl[(r - r0) * ncl + my_rank] = (unsigned char)q;
          }
        }
        named_sync(1, (uint32_t)n_deal);
        int* tmp = cur;
        cur = nxt;
        nxt = tmp;
        stale = first != last;
      }
      if (stale && nr > 0) rank_own();
      if (q < ncl && sub == 0) {
        by_rank[my_rank] = q;
        rank_of[q] = my_rank;
      }
    }
    if (pb == 0) __syncthreads();
  }
  // The leftover tiles are cut into equal pieces, at most one per cluster: tile i into
  // k_i = ceil(ns_i / T) pieces (an empty tile: one), with T the smallest piece length for
  // which the pieces fit the clusters.  T is at least kMinPiece steps and cuts no tile into
  // more than kMaxPieces pieces.  Every warp of the group tests one candidate length per
  // round (the piece count falls as the length grows), so two or three rounds find T; the
  // group's first warp then takes the prefix sums (fewer than ncl leftover tiles).
  __shared__ int s_pieces, s_slots, s_split, s_mx, s_lo, s_hi;
  __shared__ int s_fit[32];
  const int pt = (int)threadIdx.x - pb, npt = (int)blockDim.x - pb;  // multiples of 32
  if (pt >= 0) {
    if (pt == 0) s_mx = 0;
    named_sync(2, (uint32_t)npt);
    for (int i = pt; i < nr; i += npt) {
      int b, t;
      tile_at(nd + i, b, t);
      rs[i] = tile_steps(a, P_of(b), t);
      atomicMax(&s_mx, rs[i]);
    }
    named_sync(2, (uint32_t)npt);
    if (pt == 0) {
      const int mx = s_mx;
      s_lo = max(kMinPiece, (mx + kMaxPieces - 1) / kMaxPieces);
      s_hi = max(s_lo, mx);  // count(hi) <= nr < ncl: hi fits
    }
    named_sync(2, (uint32_t)npt);
    {
      const int nw = min(npt >> 5, 32), w = pt >> 5, lane = pt & 31;
      for (;;) {
        const int lo = s_lo, hi = s_hi;
        if (lo >= hi) break;
        const int stride = (hi - lo + nw - 1) / nw;
        const int len = lo + w * stride;
        if (w < nw && len < hi) {
          int c = 0;
          for (int i = lane; i < nr; i += 32) c += max(1, (rs[i] + len - 1) / len);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
          if (lane == 0) s_fit[w] = c <= ncl ? 1 : 0;
        }
        named_sync(2, (uint32_t)npt);
        if (pt < 32) {
          // candidates in increasing length: the first that fits is the new upper end, the
          // one before it (which does not) sets the new lower end
          const int l2 = lo + pt * stride;
          const uint32_t fit = __ballot_sync(0xffffffffu, pt < nw && l2 < hi && s_fit[pt]);
          if (pt == 0) {
            const int f = fit ? __ffs(fit) - 1 : -1;  // first candidate that fits
            const int tested = min(nw, (hi - lo + stride - 1) / stride);
            if (f >= 0) {
              s_lo = f > 0 ? lo + (f - 1) * stride + 1 : lo;
              s_hi = lo + f * stride;
            } else {
              s_lo = lo + (tested - 1) * stride + 1;
            }
          }
        }
        named_sync(2, (uint32_t)npt);
      }
    }
    if (pt < 32) {
      const int lane = pt;
      const int lo = s_lo;
      // k_i, first piece su[i] and first slot sbase[i] (exclusive prefix sums, 32 at a time);
      // the split tiles (k_i > 1) listed in order for the merge
      int run_c = 0, run_s = 0, run_q = 0;
      for (int i0 = 0; i0 < nr; i0 += 32) {
        const int i = i0 + lane;
        const int k = i < nr ? max(1, (rs[i] + lo - 1) / lo) : 0;
        const int ks = k > 1 ? k : 0;
        int ic = k, is = ks;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int vc = __shfl_up_sync(0xffffffffu, ic, o);
          const int vs = __shfl_up_sync(0xffffffffu, is, o);
          if (lane >= o) {
            ic += vc;
            is += vs;
          }
        }
        const uint32_t split = __ballot_sync(0xffffffffu, k > 1);
        if (i < nr) {
          su[i] = run_c + ic - k;
          sbase[i] = run_s + is - ks;
          rk[i] = k;
          if (k > 1) {
            int b, t;
            tile_at(nd + i, b, t);
            a.split_info[run_q + __popc(split & ((1u << lane) - 1u))] =
                make_int4(b, t, k, run_s + is - ks);
          }
        }
        run_c += __shfl_sync(0xffffffffu, ic, 31);
        run_s += __shfl_sync(0xffffffffu, is, 31);
        run_q += __popc(split);
      }
      if (lane == 0) {
        s_pieces = run_c;
        s_slots = run_s;
        s_split = run_q;
      }
    }
  }
  __syncthreads();
  const int n_pieces = s_pieces, n_slots = s_slots;
  if (n_slots > a.max_slots || n_pieces > ncl) {  // cannot happen (see above)
    if (threadIdx.x == 0) {
      report(a.status, TV_ERR_UNSUPPORTED);
      a.cl_start[ncl + 1] = 0;
      a.cl_start[ncl + 2] = 0;
    }
    for (int c = threadIdx.x; c <= ncl; c += blockDim.x) a.cl_start[c] = 0;
    return;
  }
  // piece k goes to cluster by_rank[k]; off[c] counts the pieces on clusters before c
  if (threadIdx.x < 32) {
    int run = 0;
    for (int c0 = 0; c0 < ncl; c0 += 32) {
      const int c = c0 + (int)threadIdx.x;
      const uint32_t m = __ballot_sync(0xffffffffu, c < ncl && rank_of[c] < n_pieces);
      if (c < ncl) off[c] = run + __popc(m & ((1u << threadIdx.x) - 1u));
      run += __popc(m);
    }
  }
  __syncthreads();
  // cluster c: its R whole tiles, then one piece if it was given one
  for (int c = threadIdx.x; c < ncl; c += blockDim.x) a.cl_start[c] = c * R + off[c];
  if (threadIdx.x == 0) {
    a.cl_start[ncl] = nd + n_pieces;
    a.cl_start[ncl + 1] = n_slots;
    a.cl_start[ncl + 2] = s_split;
  }
  // whole tiles of the first R rounds
  for (int pos = threadIdx.x; pos < nd; pos += blockDim.x) {
    const int r = pos / ncl, i = pos - r * ncl;
    const int c = r >= r0 ? (int)tcl[pos - r0 * ncl] : ((r & 1) ? ncl - 1 - i : i);
    int b, t;
    tile_at(pos, b, t);
    put(c * R + off[c] + r, b, t, 0, tile_steps(a, P_of(b), t), 1, -1, -1);
  }
  // the pieces of the leftover tiles, one thread per piece: piece k belongs to the last
  // tile i with su[i] <= k
  for (int k = (int)blockDim.x - 1 - (int)threadIdx.x; k < n_pieces; k += blockDim.x) {
    int l = 0, h = nr - 1;
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (su[m] <= k) l = m; else h = m - 1;
    }
    const int i = l, j = k - su[i], c = by_rank[k];
    int b, t;
    tile_at(nd + i, b, t);
    const int ns = rs[i], np = rk[i];
    const int s0 = j * ns / np, s1 = (j + 1) * ns / np;  // ns < 2^20, np <= kMaxPieces
    put(c * R + off[c] + R, b, t, s0, s1, np, np > 1 ? sbase[i] + j : -1,
        np > 1 ? sbase[i] : -1);
  }
}

// Merge of split tiles, after the attention kernel: one warp per row, 8 rows per work unit,
// 16 units per split tile, the units dealt to the blocks in turn (a grid of one wave, so
// that no block is launched only to find no work).  Lane k < pieces takes piece k's
// log-sum-exp; then, in slot order,
//   lse = ln sum_k exp(lse_k),  out = sum_k exp(lse_k - lse) out_k
// with four 16-byte columns per lane in flight.
__global__ void __launch_bounds__(256, 2)
merge_kernel(const int4* __restrict__ split_info, const int32_t* __restrict__ n_split,
             const float* __restrict__ ws_out, const float* __restrict__ ws_lse, int rows_seq,
             float* __restrict__ out, float* __restrict__ lse) {
  const int units = __ldg(n_split) * (kRows / 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int4 si = __ldg(split_info + u / (kRows / 8));  // {b, t, pieces, first slot}
    const int s = si.w;
    const int row = (u % (kRows / 8)) * 8 + warp;
    const int trow = si.y * kRows + row;
    if (trow >= rows_seq) continue;
    const int64_t grow = (int64_t)si.x * rows_seq + trow;
    const int np = si.z;
    const float ls = lane < np ? ws_lse[(int64_t)(s + lane) * kRows + row] : -INFINITY;
    float mx = ls;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float e = (lane < np && mx != -INFINITY && ls != -INFINITY) ? expf(ls - mx) : 0.f;
    float wsum = 0.f;
    for (int k = 0; k < np; ++k) wsum += __shfl_sync(0xffffffffu, e, k);
    const float w = wsum > 0.f ? e / wsum : 0.f;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    // four pieces' loads in flight at a time (a piece at a time left the warp waiting on
    // one memory round trip per piece); the products are summed in piece order as before
    for (int k0 = 0; k0 < np; k0 += 4) {
      float wk[4];
      float4 v[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int k = k0 + q;
        wk[q] = __shfl_sync(0xffffffffu, w, k < np ? k : 0);
        if (k >= np) wk[q] = 0.f;
        if (wk[q] != 0.f) {  // the same for the whole warp
          const float4* src =
              reinterpret_cast<const float4*>(ws_out + ((int64_t)(s + k) * kRows + row) * kDL);
#pragma unroll
          for (int i = 0; i < 4; ++i) v[q][i] = __ldcs(src + lane + 32 * i);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) v[q][i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (wk[q] == 0.f) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i].x = fmaf(wk[q], v[q][i].x, acc[i].x);
          acc[i].y = fmaf(wk[q], v[q][i].y, acc[i].y);
          acc[i].z = fmaf(wk[q], v[q][i].z, acc[i].z);
          acc[i].w = fmaf(wk[q], v[q][i].w, acc[i].w);
        }
      }
    }
    float4* d4 = reinterpret_cast<float4*>(out + grow * kDL);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[lane + 32 * i] = acc[i];
    if (lane == 0) lse[grow] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
  }
}

// Work preparation, one launch before the attention kernel.
//  - Block 0 writes the work schedule (schedule(), above).
//  - Paged cache: the other blocks write, for every 128-key step of every sequence, the
//    step's two tensor maps (latent and rope).  Each is a copy of a host-encoded template
//    with a new base (the step's lower page), page-dimension stride (distance to its other
//    page; 0 if both are the same page) and, when the step has one page only, page extent
//    1 (the missing half reads as zeros).  The fields are edited on a copy in shared
//    memory (edits of a map in global memory are slow read-modify-writes, and a thread
//    makes six of them), which is then stored to global memory.  A page index outside the
//    cache rows is reported as TV_ERR_BOUNDS and replaced by page 0 (that sequence's result
//    is then undefined, as for any out-of-range input).
__device__ __forceinline__ void prep_body(
    const SchedArgs& sa, const CUtensorMap& tmpl_lat, const CUtensorMap& tmpl_rope,
    const unsigned char* ckv, int64_t ckv_page_bytes, const unsigned char* kpe,
    int64_t kpe_page_bytes, const int32_t* __restrict__ page_table, int max_pages,
    int64_t num_pages, int steps_per_seq, CUtensorMap* __restrict__ maps,
    uint8_t* __restrict__ swap, unsigned char* buf) {
  const int32_t* prefix_len = sa.prefix_len;
  const int B = sa.B, Q = sa.Q, max_prefix = sa.max_prefix;
  const int64_t seq_cap = sa.seq_cap;
  int32_t* status = sa.status;
  if (blockIdx.x > 0) {
    if (threadIdx.x >= kMapThreads) return;
    const int64_t idx = (int64_t)(blockIdx.x - 1) * kMapThreads + threadIdx.x;
    if (idx >= (int64_t)B * steps_per_seq) return;
    const int b = (int)(idx / steps_per_seq), sp = (int)(idx - (int64_t)b * steps_per_seq);
    const int P = prefix_len[b];
    const int64_t kv = (int64_t)P + Q;
    if (P < 0 || P > max_prefix || kv > seq_cap) return;  // reported by the attention kernel
    const int64_t nblk = (kv + kBN - 1) / kBN;
    if (2 * (int64_t)sp >= nblk) return;  // beyond this sequence: never used
    int64_t pa = page_table[(int64_t)b * max_pages + 2 * sp];
    const bool has_b = 2 * (int64_t)sp + 1 < nblk;
    int64_t pb = has_b ? page_table[(int64_t)b * max_pages + 2 * sp + 1] : pa;
    if (pa < 0 || pa >= num_pages || pb < 0 || pb >= num_pages) {
      report(status, TV_ERR_BOUNDS);
      pa = pb = 0;
    }
    const int64_t lo = pa < pb ? pa : pb, dist = pa < pb ? pb - pa : pa - pb;
    uint4* sl = reinterpret_cast<uint4*>(buf + threadIdx.x * 256);
    uint4* sr = sl + 8;
    const uint4* tl = reinterpret_cast<const uint4*>(&tmpl_lat);
    const uint4* tr = reinterpret_cast<const uint4*>(&tmpl_rope);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      sl[w] = tl[w];
      sr[w] = tr[w];
    }
    const uint32_t al = smem_u32(sl), ar = smem_u32(sr);
    tmap_set_address_smem(al, ckv + lo * ckv_page_bytes);
    tmap_set_stride2_smem(al, (uint64_t)(dist * ckv_page_bytes));
    tmap_set_address_smem(ar, kpe + lo * kpe_page_bytes);
    tmap_set_stride2_smem(ar, (uint64_t)(dist * kpe_page_bytes));
    if (!has_b) {
      tmap_set_dim3_smem(al, 1);
      tmap_set_dim3_smem(ar, 1);
    }
    uint4* ml = reinterpret_cast<uint4*>(maps + 2 * idx);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      ml[w] = sl[w];
      ml[8 + w] = sr[w];
    }
    swap[idx] = (uint8_t)(pb < pa ? 1 : 0);
    tmap_release();
    return;
  }
  schedule(sa, buf);
}

// overlap = 0: launched in stream order.  overlap = 1 (tv_attn_args.overlap_prev): launched
// as a programmatic dependent of the kernel before it, whose outputs it does not read; it
// does its work while that kernel finishes and waits for it only before leaving, so that
// the attention kernel's wait on this grid covers both.
__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(const SchedArgs sa, const __grid_constant__ CUtensorMap tmpl_lat,
            const __grid_constant__ CUtensorMap tmpl_rope, const unsigned char* ckv,
            int64_t ckv_page_bytes, const unsigned char* kpe, int64_t kpe_page_bytes,
            const int32_t* __restrict__ page_table, int max_pages, int64_t num_pages,
            int steps_per_seq, CUtensorMap* __restrict__ maps, uint8_t* __restrict__ swap,
            int overlap) {
  __shared__ __align__(128) unsigned char buf[kPrepSmem];
  griddep_launch_dependents();  // the attention kernel may start its set-up now
  prep_body(sa, tmpl_lat, tmpl_rope, ckv, ckv_page_bytes, kpe, kpe_page_bytes, page_table,
            max_pages, num_pages, steps_per_seq, maps, swap, buf);
  if (overlap) griddep_wait();
}

// ---- host side -----------------------------------------------------------------------
// Testing hook (tv_testing_set_wait_fault): off unless a test turns it on.
std::mutex g_test_mu;
int g_test_skip_loads = 0;
uint64_t g_test_deadline_ns = 0;
int32_t* g_test_exit_counts = nullptr;

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

// Latent rows viewed as [64 elements][rows][8 chunks of 64 elements]: one box is
// `box_chunks` chunks of `box_rows` rows, landing chunk-major in shared memory as
// 128-byte-swizzled tiles.
bool make_map_latent(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes,
                     uint32_t box_rows, uint32_t box_chunks) {
  cuuint64_t dims[3] = {64, rows, kDL / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rope rows: one box is 64 elements of `box_rows` rows.
bool make_map_rope(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes,
                   uint32_t box_rows) {
  cuuint64_t dims[2] = {kDR, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {64, box_rows};
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
                             kSmemBytes) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
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

// Rows per sequence of a gathered key view: the longest KV rounded up to whole steps.
int64_t gathered_seq_rows(const tv_attn_args* a) {
  const int64_t kv_max = (int64_t)a->max_prefix_len + a->Q;
  return (kv_max + kStep - 1) / kStep * kStep;
}

// Paged cache: gather it into a contiguous view (true) or use per-step tensor maps (false).
// AUTO uses the per-step maps: on the B32 Q33 workload they now run the attention call at
// least as fast as the gathered view (0.831 vs 0.839 ms) without its extra copy of the keys
// (about 450 MB of HBM traffic and a 300 MB workspace).  TV_PAGED_GATHER forces the copy.
bool use_gather(const tv_attn_args* a) {
  if (!a->cache.page_table || a->paged_view != TV_PAGED_GATHER) return false;
  const int64_t rows = (int64_t)a->B * gathered_seq_rows(a);
  return rows < (1ll << 31);
}

// 128-key steps of the longest sequence (per-step tensor maps of a paged cache).
int64_t steps_per_seq(const tv_attn_args* a) {
  return ((int64_t)a->max_prefix_len + a->Q + kStep - 1) / kStep;
}

// Templates of the per-step maps of a paged cache.  Latent: {64 elements, 8 rows, 8 row
// groups, 2 pages, 8 chunks} with strides {row, 8 rows, page placeholder, 128 bytes}, box
// {64, 8, 8, 2, 2} (two chunks of 128 keys, the same shared-memory layout as a 3-D box of
// 128 consecutive rows).  Rope: {64 elements, 8 rows, 8 row groups, 2 pages}, box = all.
bool make_step_templates(CUtensorMap* lat, CUtensorMap* rope, const tv_attn_args* a) {
  const uint64_t rb = (uint64_t)a->ckv_row_stride * 2, rbk = (uint64_t)a->kpe_row_stride * 2;
  {
    cuuint64_t dims[5] = {64, 8, 8, 2, kDL / 64};
    cuuint64_t strides[4] = {rb, 8 * rb, 64 * rb, 128};
    cuuint32_t box[5] = {64, 8, 8, 2, 2};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (g_encode(lat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(a->c_kv), dims, strides,
                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  cuuint64_t dims[4] = {kDR, 8, 8, 2};
  cuuint64_t strides[3] = {rbk, 8 * rbk, 64 * rbk};
  cuuint32_t box[4] = {64, 8, 8, 2};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return g_encode(rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a->k_pe), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

bool tc_supported(const tv_attn_args* a) {
  if (!(a->q_dt == TV_BF16 && a->kv_dt == TV_BF16 && a->d_latent == kDL && a->d_rope == kDR &&
        a->cache.num_rows > 0 && a->cache.num_rows < (1ll << 31)))
    return false;
  return a->cache.page_table == nullptr || a->cache.page_size == kBN;
}

TcPlan tc_plan(const tv_attn_args* a) {
  TcPlan p{};
  const int clusters = max_clusters() > 0 ? max_clusters() : 74;
  p.clusters = std::min(clusters, kMaxSchedClusters);
  p.tiles_per_seq = (a->Q * a->H + kRows - 1) / kRows;
  p.n_tiles = (int64_t)a->B * p.tiles_per_seq;
  p.splits = a->num_splits > 0 ? std::min(a->num_splits, kMaxForcedSplits) : 0;
  if (p.splits > 0) {
    p.n_items = p.n_tiles * p.splits;
    p.max_slots = p.splits > 1 ? p.n_items : 0;
    p.max_split = p.splits > 1 ? p.n_tiles : 0;
  } else {
    // whole tiles, plus at most one piece per cluster (slots: twice that, a loose bound)
    p.n_items = p.n_tiles + p.clusters;
    p.max_slots = 2 * (int64_t)p.clusters;
    p.max_split = p.clusters;  // split tiles are among the fewer than `clusters` left over
  }
  return p;
}

// Workspace: [item records: 32 B each][cluster list starts, then the item, slot and
// split-tile counts][slot records][split-tile records][partial outputs: slot x 128 x 512
// fp32][partial lse][paged
// cache: gathered key view, or per-step tensor maps (2 x 128 B per step) and swap flags].
struct TcWs {
  size_t items, cl_start, slot_info, split_info, part_out, part_lse, tail, total;
};
TcWs tc_ws_layout(const tv_attn_args* a, const TcPlan& p) {
  TcWs w{};
  size_t n = 0;
  w.items = n;
  n += align256((size_t)p.n_items * 32);
  w.cl_start = n;
  n += align256(((size_t)p.clusters + 3) * 4);
  w.slot_info = n;
  n += align256((size_t)p.max_slots * 16);
  w.split_info = n;
  n += align256((size_t)p.max_split * 16);
  w.part_out = n;
  n += align256((size_t)p.max_slots * kRows * kDL * 4);
  w.part_lse = n;
  n += align256((size_t)p.max_slots * kRows * 4);
  w.tail = n;
  if (use_gather(a)) {
    n += align256((size_t)a->B * (size_t)gathered_seq_rows(a) * (kDL + kDR) * 2);
  } else if (a->cache.page_table) {
    const size_t steps = (size_t)a->B * (size_t)steps_per_seq(a);
    n += align256(steps * 2 * sizeof(CUtensorMap)) + align256(steps);
  }
  w.total = n;
  return w;
}

size_t tc_workspace(const tv_attn_args* a, const TcPlan& p) { return tc_ws_layout(a, p).total; }

int tc_launch_count(const tv_attn_args* a, const TcPlan& p) {
  return 2 + (use_gather(a) ? 1 : 0) + (p.max_slots > 0 ? 1 : 0);
}

cudaError_t launch_attn_tc(const tv_attn_args* a, const TcPlan& pl, void* ws, cudaStream_t st) {
  if (!get_encode()) return cudaErrorNotSupported;
  if (max_clusters() <= 0) return cudaErrorNotSupported;
  const size_t rows = (size_t)a->B * a->Q * a->H;
  const TcWs lay = tc_ws_layout(a, pl);
  char* const ws0 = (char*)ws;
  char* wsp = ws0 + lay.tail;
  const bool gather = use_gather(a);
  const bool paged = a->cache.page_table != nullptr && !gather;  // per-step maps
  const int64_t steps = paged ? steps_per_seq(a) : 0;
  CUtensorMap* maps = nullptr;
  uint8_t* swap = nullptr;
  if (paged) {
    maps = (CUtensorMap*)wsp;
    wsp += align256((size_t)a->B * steps * 2 * sizeof(CUtensorMap));
    swap = (uint8_t*)wsp;
  }
  // the key view the attention kernel reads rows of: the cache, or its gathered copy
  int64_t seq_rows, seq_cap;
  uint64_t key_rows, lat_row_bytes, kpe_row_bytes;
  const void* lat_base;
  const void* kpe_base;
  if (gather) {
    seq_rows = gathered_seq_rows(a);
    seq_cap = std::min<int64_t>(seq_rows, (int64_t)a->cache.max_pages * kBN);
    key_rows = (uint64_t)a->B * (uint64_t)seq_rows;
    lat_base = wsp;
    kpe_base = wsp + kDL * 2;
    lat_row_bytes = kpe_row_bytes = (kDL + kDR) * 2;
  } else {
    seq_rows = paged ? 0 : a->cache.kv_stride_b;
    seq_cap = paged ? (int64_t)a->cache.max_pages * kBN : a->cache.kv_stride_b;
    key_rows = (uint64_t)a->cache.num_rows;
    lat_base = a->c_kv;
    kpe_base = a->k_pe;
    lat_row_bytes = (uint64_t)a->ckv_row_stride * 2;
    kpe_row_bytes = (uint64_t)a->kpe_row_stride * 2;
  }
  // S-side maps over the row view (unused with per-step maps) and the O-side map
  CUtensorMap m_lat_s, m_kpe_s, m_lat_o, t_lat, t_rope;
  if (!make_map_latent(&m_lat_s, lat_base, key_rows, lat_row_bytes, kStep, 2) ||
      !make_map_rope(&m_kpe_s, kpe_base, key_rows, kpe_row_bytes, kStep) ||
      !make_map_latent(&m_lat_o, lat_base, key_rows, lat_row_bytes, kBN, 4))
    return cudaErrorInvalidValue;
  if (paged && !make_step_templates(&t_lat, &t_rope, a)) return cudaErrorInvalidValue;
  // query tiles: 128 rows of latent queries as four {64, 128, 2} boxes, rope queries as one
  // {64, 128} box (rows past the last one read zeros)
  CUtensorMap m_q, m_qr;
  if (!make_map_latent(&m_q, a->q_latent, (uint64_t)rows, kDL * 2, kRows, 2) ||
      !make_map_rope(&m_qr, a->q_pe, (uint64_t)rows, kDR * 2, kRows))
    return cudaErrorInvalidValue;
  if (!paged) {
    t_lat = m_lat_s;  // not used
    t_rope = m_kpe_s;
  }

  TcParams p{};
  p.q_latent = (const __nv_bfloat16*)a->q_latent;
  p.q_pe = (const __nv_bfloat16*)a->q_pe;
  p.seq_rows = seq_rows;
  p.seq_cap = seq_cap;
  p.prefix_len = a->prefix_len;
  p.anc = a->anc;
  p.out = a->out;
  p.lse = a->lse;
  p.ws_out = (float*)(ws0 + lay.part_out);
  p.ws_lse = (float*)(ws0 + lay.part_lse);

  p.status = a->status;
  p.rows_total = (int64_t)rows;
  p.B = a->B;
  p.H = a->H;
  p.Q = a->Q;
  p.max_prefix = a->max_prefix_len;
  p.tiles_per_seq = pl.tiles_per_seq;
  p.items = (const int4*)(ws0 + lay.items);
  p.cl_start = (const int32_t*)(ws0 + lay.cl_start);
  p.step_maps = maps;
  p.step_swap = swap;
  p.page_table = a->cache.page_table;
  p.steps_per_seq = (int32_t)steps;
  p.max_pages = a->cache.max_pages;
  p.paged = paged ? 1 : 0;
  p.scale_log2 = (float)((double)a->scale * 1.4426950408889634);
  p.timeout_ns = kTimeoutNs;
  p.causal = a->mask_mode == TV_MASK_CAUSAL ? 1 : 0;
  {
    std::lock_guard<std::mutex> lock(g_test_mu);
    p.test_skip_loads = g_test_skip_loads;
    if (g_test_deadline_ns) p.timeout_ns = g_test_deadline_ns;
    p.test_exit_counts = g_test_exit_counts;
  }
  if (pl.n_tiles == 0) return cudaSuccess;
  // clusters launched: all of them (the schedule spreads the work over all), or with
  // forced splits no more than there are items
  const int ncl = (int)std::min<int64_t>(pl.clusters, pl.splits > 0 ? pl.n_items : pl.clusters);

  {
    SchedArgs sa{};
    sa.prefix_len = a->prefix_len;
    sa.B = a->B;
    sa.Q = a->Q;
    sa.H = a->H;
    sa.T = pl.tiles_per_seq;
    sa.causal = p.causal;
    sa.max_prefix = a->max_prefix_len;
    sa.seq_cap = seq_cap;
    sa.ncl = ncl;
    sa.splits = pl.splits;
    sa.max_slots = (int)pl.max_slots;
    sa.items = (int4*)(ws0 + lay.items);
    sa.cl_start = (int32_t*)(ws0 + lay.cl_start);
    sa.slot_info = (int4*)(ws0 + lay.slot_info);
    sa.split_info = (int4*)(ws0 + lay.split_info);
    sa.status = a->status;
    const int64_t map_blocks = paged ? (a->B * steps + kMapThreads - 1) / kMapThreads : 0;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((unsigned)(1 + map_blocks));
    pc.blockDim = dim3(kPrepThreads);
    pc.stream = st;
    cudaLaunchAttribute pat[1];
    pat[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pat[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pat;
    pc.numAttrs = a->overlap_prev ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(
        &pc, prep_kernel, sa, t_lat, t_rope, (const unsigned char*)a->c_kv,
        (int64_t)lat_row_bytes * kBN, (const unsigned char*)a->k_pe, (int64_t)kpe_row_bytes * kBN,
        a->cache.page_table, a->cache.max_pages, (int64_t)a->cache.num_rows / kBN, (int)steps,
        maps, swap, a->overlap_prev ? 1 : 0);
    if (e != cudaSuccess) return e;
  }
  if (gather) {
    const dim3 grid((unsigned)(seq_rows / kBN), (unsigned)a->B);
    gather_kv_kernel<<<grid, 256, 0, st>>>(
        (const uint4*)a->c_kv, a->ckv_row_stride / 8, (const uint4*)a->k_pe, a->kpe_row_stride / 8,
        a->cache.page_table, a->cache.max_pages, a->prefix_len, a->Q, a->max_prefix_len,
        a->cache.num_rows, seq_rows, (uint4*)wsp, a->status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ncl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tc_kernel, p, m_lat_s, m_kpe_s, m_lat_o, m_q, m_qr);
  if (e != cudaSuccess || pl.max_slots == 0) return e;
  // merge the pieces of split tiles: two blocks per SM (one wave at the merge's register
  // count), or fewer when there cannot be that many units of work
  const int64_t merge_blocks =
      std::min<int64_t>(pl.max_split * (kRows / 8), 4 * (int64_t)pl.clusters);
  merge_kernel<<<(unsigned)merge_blocks, 256, 0, st>>>(
      (const int4*)(ws0 + lay.split_info), (const int32_t*)(ws0 + lay.cl_start) + ncl + 2,
      p.ws_out, p.ws_lse, a->Q * a->H, a->out, a->lse);
  return cudaGetLastError();
}

}  // namespace tv

extern "C" int tv_testing_set_wait_fault(int skip_key_loads, uint64_t deadline_ns,
                                         int32_t* exit_counts) {
  if (skip_key_loads < 0 || skip_key_loads > 1) return TV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(tv::g_test_mu);
  tv::g_test_skip_loads = skip_key_loads;
  tv::g_test_deadline_ns = deadline_ns;
  tv::g_test_exit_counts = exit_counts;
  return TV_OK;
}
