// Streaming path of the delayed mHC seam: bandwidth-tuned for large T, and
// latency-tuned for small T with larger clusters.
//
// Persistent clusters of KCL CTAs (4, or 16 for small T; one CTA per SM).
// CTA r of a cluster owns the 64-column chunks r, r + KCL, r + 2 KCL, ... of H
// for all four streams (the cluster reads each row in long runs) and the
// cluster walks blocks of 32 tokens (its items: blocks cid, cid + ncl, ...,
// or blocks taken by ticket; see SCHED below).  Per 64-column chunk:
//  - an input producer warp TMA-loads the four R tiles and the Y tile into a
//    ring of 4 input stages (5 without Y; 128-byte swizzle), and, during each
//    item, the next item's carried gates (comb, pre, post) into one of two
//    buffers, so they wait in shared memory when compute gets there;
//  - an fn producer warp TMA-loads the four hi/lo-packed fn tiles [48 x 64]
//    into a ring of 2 fn stages (L2 evict-last: every cluster reuses them);
//  - eight compute warps (thread = token, warp = 8-column slice; the swizzle
//    makes the column reads conflict-free) read their inputs, release the
//    input stage, post-mix in fp32 (packed fp32x2 FMAs), round R' to bf16 into
//    a ring of 3 output stages, accumulate s_R and s_x, keep x in tensor
//    memory, and normalise the previous block's x of the same chunk into the
//    same output stage;
//  - the gate projection runs on the tensor cores, in one of two forms:
//    tcgen05 (one thread issues 4 MMAs per chunk: A = the four R' tiles
//    stacked [128 x 64], B = the four fn tiles side by side [192 x 64], so
//    D[128 x 192] holds stream i's 32 x 48 block on its diagonal, in TMEM
//    lanes 32 i.. and columns 48 i..; the off-diagonal products are wasted,
//    but each MMA instruction costs the same whatever its size), or, where x
//    leaves no room for that accumulator in tensor memory, warp-level m16n8k16
//    MMAs in the compute warps;
//  - a store warp TMA-stores the R' tiles and the norm tile of each stage
//    (and computes the e4m3 codes and ue8m0 scales of the norm tile); with
//    the fp8_grid output three more warps each take every third stage and
//    write the grid of its norm tile.
// After the last chunk of a block the compute warps hand their partial sums
// over in shared memory and go on; an exchange warp sends, through
// distributed shared memory (st.async completing bytes on the receiver's
// mbarrier):
//  - the CTA's per-token s_x partials to every CTA of the cluster, which each
//    sum them in the same order into rstd_x, needed by the next block's first
//    chunk;
//  - the 24 projection sums and s_R of each token to the token's owner CTA
//    (token % KCL), whose exchange warp then computes the gates.
// With the split schedule the blocks of the partial last round are cut into
// column parts whose partial sums meet in a global workspace instead.
// ("[FlyDSL] Single-launch Mega-mHC on gfx950", Kernel Architecture: split-K
// with a distributed finish; here the cluster launch makes every CTA of a
// split co-resident.)
//
// Forms: post, no_post, and identity (the first block's seam: R' = R, no
// residual store).  A call with no norm pointer stores no norm: the first
// pass of the unshifted ordering, which needs only R' and the gates.
//
// Every wait is bounded, in two tiers.  A wait longer than the caller's limit
// flags the CTA (the kernel's exit sets bit 1 of the status word) and goes on
// waiting, so a short limit only flags the call and the work completes as
// usual.  A wait one second longer
// abandons the call: the CTA stops issuing copies, MMAs and stores, and before
// it frees tensor memory and exits it waits (with a fixed cap) for the ones in
// flight: the last TMA load of every input, fn and gate buffer (a buffer is
// refilled only after its previous load was seen complete), every MMA (one
// final tcgen05.commit) and every bulk store (bulk wait_group).

#pragma once

#include "mhc_common.cuh"
#include "mhc_sm100.cuh"

namespace mhc {

namespace {

constexpr int kBM = 32;                // tokens per block
constexpr int kChunk = 64;             // columns per chunk
constexpr int kNF = 2, kNO = 3;
// warps 0-7 compute, 8 input producer, 9 MMA issuer, 10 fn producer, 11 finisher, 12 store,
// and with the fp8_grid output 13-15 grid warps (warp 13 + o takes output
// stage o).  16 warps still leave each thread 128 registers (4 warps per SM
// sub-partition, as with 13).
template <int OUT>
__host__ __device__ constexpr int threads_of() { return OUT == 2 ? 512 : 416; }
constexpr int kFnRows = 48;
constexpr uint32_t kRTile = kBM * 128;                 // 4 KB
constexpr uint32_t kFnTile = kFnRows * 128;            // 6 KB
constexpr uint32_t kFnStage = 4 * kFnTile;             // 24 KB: [192 x 64] bf16
constexpr uint32_t kInStage = 5 * kRTile;              // 20 KB: R tiles 0-3, Y tile 4
// The input ring of clusters of 4 holds 4 stages of R + Y, or, in the forms
// without Y, 5 stages of R in the same bytes (more loads in flight per SM);
// clusters of 16 (a CTA has at most 8 chunks per block) hold 3 stages.
constexpr int kNIMax = 8;
template <int FORM, int KCL>
__host__ __device__ constexpr int in_stages() { return KCL == 16 ? 3 : FORM == 1 ? 4 : 5; }
template <int FORM>
__host__ __device__ constexpr uint32_t in_stage_bytes() { return FORM == 1 ? kInStage : 4 * kRTile; }
constexpr uint32_t kOffNormT = 4 * kRTile;             // output stage: R' tiles 0-3, then the norm tile,
constexpr uint32_t kOffCodesT = 5 * kRTile;            //   then (mxfp8) the codes tile [32 x 64] u8
// 22 KB with the codes tile, else 20 KB (multiples of 1 KB: swizzled tiles)
template <int OUT>
__host__ __device__ constexpr uint32_t out_stage_bytes() { return OUT == 1 ? 5 * kRTile + kBM * 64 : 5 * kRTile; }
// The normalise-only pass after a cluster's last block puts the norm tiles of
// norm_group() chunks in one output stage (in the R' tile slots; with mxfp8
// the codes tiles go where the norm tile sits in the other passes).
template <int OUT>
__host__ __device__ constexpr int norm_group() { return OUT == 1 ? 2 : 4; }
constexpr uint32_t kOffFn = 0;
constexpr uint32_t kOffOut = kOffFn + kNF * kFnStage;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;                          // tcgen05 accumulator D[128 x 192]
constexpr uint32_t kDCols = 4 * kFnRows;
constexpr int kMaxChunksTC = (int)((kTmemCols - kDCols) / 16);  // x: 16 columns per chunk
constexpr int kMaxChunks = (int)(kTmemCols / 16);
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kDCols);
constexpr int kOwnerParts = 25;                        // sent to a token's owner: 24 projections, s_R
constexpr int kPartPad = 26;                           // rows of 8-byte aligned pairs
constexpr int kDPad = 25;                              // odd row stride: conflict-free columns

// Carried gates of one block, TMA-loaded a block ahead: comb [32 x 16],
// pre [32 x 4], post [32 x 4] fp32.
struct alignas(128) GateTile {
  float comb[kBM][16];
  float pre[kBM][4];
  float post[kBM][4];
};

// One item of a cluster's work as its rank-0 CTA publishes it (see the
// schedule below).
struct alignas(16) Item {
  int block;  // token block of 32 tokens; -1: the cluster's list has ended; -2: the call was abandoned
  int g0;     // first column group
  int ng;     // column groups (all G for a whole block)
  int unit;   // unit id v (index of its global partial sums), -1 for a whole block
};
constexpr int kSchedD = 4;         // items published ahead and not yet read by every CTA
constexpr int kMaxUnitsCl = 16;    // units one cluster may hold

// Geometry of a cluster of KCL CTAs: 4 for large T (bandwidth), 16 for small T
// (each CTA takes a quarter of the columns it would take in a cluster of 4),
// for output mode OUT (the mxfp8 output stages hold a codes tile more).
// LEAN: the identity form with the tcgen05 projection, whose MMAs read
// R' = R from the input stage: an output stage then holds only the norm tile
// (and the codes tile), and the shared memory this frees goes to the input
// ring (8 stages of R instead of 5 on clusters of 4: more loads in flight per
// SM, which is what bounds that form).
template <int KCL, int OUT, bool LEAN = false>
struct Geo {
  static constexpr int kCl = KCL;
  static constexpr uint32_t kOutStage = LEAN ? (OUT == 1 ? kRTile + kBM * 64 : kRTile) : out_stage_bytes<OUT>();
  static constexpr uint32_t kInRing = (KCL == 16 ? 3 : 4) * kInStage  // input ring: 80 KB (60 KB)
                                      + (LEAN ? kNO * (out_stage_bytes<OUT>() - kOutStage) : 0);
  // LEAN: input stages of R alone (16 KB) that fit the ring
  static constexpr int kNILean = (int)(kInRing / (4 * kRTile)) < kNIMax ? (int)(kInRing / (4 * kRTile)) : kNIMax;
  static constexpr uint32_t kOffNormT = LEAN ? 0 : 4 * kRTile;   // the norm tile in an output stage
  static constexpr uint32_t kOffCodesT = LEAN ? kRTile : 5 * kRTile;  // (mxfp8) the codes tile [32 x 64] u8
  // the normalise-only pass: norm tiles of kNormGroup chunks per stage (in
  // the R' tile slots), the codes tiles from kPassCodes on
  static constexpr int kNormGroup = LEAN ? 1 : norm_group<OUT>();
  static constexpr uint32_t kPassCodes = LEAN ? kRTile : 4 * kRTile;
  static constexpr int kSlots = kBM / KCL;              // tokens owned per CTA and block
  // gamma of a CTA's first chunks, staged in shared memory (the mxfp8 form on
  // clusters of 4 has no room left: its chunks read gamma through L1/L2)
  static constexpr int kGamChunks = KCL == 4 ? (OUT == 1 ? 0 : kMaxChunksTC) : (kMaxChunks * 4) / KCL;
  static constexpr uint32_t kXsBytes = KCL * kBM * 4;   // s_x partials landing in each CTA per block
  static constexpr uint32_t kRecvBytes = KCL * kSlots * kOwnerParts * 4;  // owner partials per CTA per block
  static constexpr uint32_t kOffIn = kOffOut + kNO * kOutStage;
  static constexpr uint32_t kOffTail = kOffIn + kInRing;
  static_assert(kOffTail % 128 == 0, "tail alignment (16-byte st.async targets, 8-byte barriers)");
  struct Tail {
    GateTile gates[2];                     // carried gates of items i (buffer i % 2), loaded an item ahead; a
                                           // buffer is released only when its item's compute has finished
    uint64_t in_full[kNIMax], in_empty[kNIMax], fn_full[kNF], fn_empty[kNF], out_full[kNO], out_empty[kNO];
    uint64_t d_full, xs_full[2], recv_full[2], recv_free[2], gates_full[2], gates_empty[2];
    uint64_t red_full[2], dbuf_full, dbuf_free, d_free;
    uint64_t red_free[2];                  // the exchange warp has read a parity's partials
    uint64_t sched_full[kSchedD];          // an item has landed in the slot (16 bytes from rank 0)
    uint64_t sched_free[kSchedD];          // (rank 0) every reader of the cluster has read the slot
    Item sched[kSchedD];                   // the cluster's items, published by rank 0
    Item ulist[kMaxUnitsCl];               // the cluster's units, in order (written by the input producer)
    int nunits;
    uint64_t mma_fin;                      // exit drain: completion of every MMA issued
    uint64_t fold_full;                    // warp-MMA form: warps 4-7 have written their partial projections
    uint32_t tmem_base;
    volatile int reported, aborted;
    float2 red[2][8][kBM];                 // [block parity][compute warp][token]: s_R, s_x partials
    float dbuf[4][kBM][kDPad];             // the block's projection per stream (hi + lo): [stream][token][logit]
    float xs[2][KCL][kBM];                 // [block parity][source CTA][token]: s_x partial
    float recv[2][KCL][kSlots][kPartPad];  // [block parity][source CTA][owned token][part]
    uint4 gam[kGamChunks > 0 ? kGamChunks : 1][8];  // gamma of this CTA's first chunks (8 bf16 per compute warp)
    float pbuf[kSlots][kPartPad];          // the owned tokens' parts summed over the cluster
    float ab[27];                          // alpha[3], bias[24]
  };
  static constexpr size_t kSmemBytes = kOffTail + sizeof(Tail) + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory of the streaming kernel exceeds 227 KB");
};

struct Ctx {
  const SeamArgs* a;
  volatile int* reported;  // the CTA has set the status bit of a slow wait
  volatile int* aborted;   // the CTA abandons the call: no new copies, MMAs or stores
  uint64_t report_ns;      // a wait longer than this is reported (status bit 1) and goes on
  uint64_t abort_ns;       // a wait longer than this abandons the call
};

// Fixed cap of the exit drain (waits for copies and MMAs this CTA issued,
// which complete on their own); independent of the caller's limit and of any
// earlier error.
constexpr uint64_t kDrainNs = 200000000ull;

// One check of a barrier wait whose phase was not complete at the first
// test (called between suspending tries of about 20 us each).  Past
// report_ns the CTA flags the call (the kernel's exit sets status bit 1) and
// the wait goes on, so a short limit only flags the call; past abort_ns, or
// at once once the CTA has abandoned the call, it returns true and the caller
// stops issuing work (it never arrives on a barrier whose phase it did not
// see complete).  Only CTA-local flags are touched, so each wait site stays
// a few instructions: the kernel's instruction footprint is what keeps its
// hot loops in the instruction cache.
__device__ __forceinline__ bool wait_gave_up(const Ctx& x, uint64_t& t0) {
  const uint64_t now = globaltimer_ns();
  if (t0 == 0) t0 = now;
  const uint64_t dt = now - t0;
  if (dt > x.report_ns) *x.reported = 1;
  if (dt > x.abort_ns || *x.aborted) {
    *x.aborted = 1;
    return true;
  }
  return false;
}
// Wait on a phase of a CTA-local barrier: a test, then suspending tries (the
// warp sleeps until the phase completes, up to about 20 us a try), each
// followed by the check above.
__device__ __forceinline__ bool wait_local(const Ctx& x, uint64_t* bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  while (!mbar_try_wait(bar, parity, 20000))
    if (wait_gave_up(x, t0)) return false;
  return true;
}
// The same on a barrier that cluster peers arrive on (acquire at cluster scope).
__device__ __forceinline__ bool wait_remote(const Ctx& x, uint64_t* bar, uint32_t parity) {
  uint64_t t0 = 0;
  while (!mbar_try_wait_cluster(bar, parity, 20000))
    if (wait_gave_up(x, t0)) return false;
  return true;
}
// A wait every lane of a warp makes: the warp goes on only if all lanes saw
// the phase complete, so the warp leaves its loop as one.
__device__ __forceinline__ bool wait_warp(const Ctx& x, uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_local(x, bar, parity));
}
__device__ __forceinline__ bool wait_warp_remote(const Ctx& x, uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_remote(x, bar, parity));
}
// Exit drain: wait for the phase that a copy or MMA this CTA issued
// completes, at most kDrainNs, whatever happened before.
__device__ __forceinline__ void drain(const Ctx& x, uint64_t* bar, uint32_t parity) {
  if (!mbar_wait(bar, parity, kDrainNs)) *x.reported = 1;
}

}  // namespace

// The fp8_grid row of one token (lane = token) and 64 columns: the row of
// the 128-byte-swizzled norm tile nt (64 bf16) into registers, then `rel`
// (if given) is arrived on by lane 0 once the warp has read the tile, then
// the bf16 of the dequantised e4m3 codes of each 32-group to dst (nullptr: a
// token past T), 128 contiguous bytes written by this thread.  Out of line
// (one copy for both call sites, the grid warps hold few live values); the
// row stays in registers (constant indices only).
static __device__ __noinline__ void grid_tile_row(const uint8_t* nt, uint64_t* rel, __nv_bfloat16* dst,
                                                  float amax_floor, int lane) {
  uint32_t nb[32];
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const uint4 v = *reinterpret_cast<const uint4*>(nt + lane * 128 + ((ch ^ (lane & 7)) << 4));
    nb[4 * ch] = v.x; nb[4 * ch + 1] = v.y; nb[4 * ch + 2] = v.z; nb[4 * ch + 3] = v.w;
  }
  __syncwarp();
  if (rel != nullptr && lane == 0) mbar_arrive(rel);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t gw[16];
    grid_group32(nb + 16 * half, gw, amax_floor);
    if (dst != nullptr) {
      uint4* d = reinterpret_cast<uint4*>(dst + 32 * half);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) st_stream(d + ch, make_uint4(gw[4 * ch], gw[4 * ch + 1], gw[4 * ch + 2], gw[4 * ch + 3]));
    }
  }
}

// Gate finish of one token on its owner CTA, kept out of line so its arrays
// do not raise the register pressure of the kernel.
static __device__ __noinline__ void finish_store_gates(const SeamArgs& a, int64_t t, const float* p, const float* ab, int H) {
  float pre[4], post[4], cb[16];
  finish_gates(p[24], p, ab, ab + 3, kStreams * H, a.eps, a.sinkhorn_iters, pre, post, cb);
  store_gates(a, t, pre, post, cb);
}

namespace {

// What one cluster works on, in order ("items"), handed out as the clusters
// ask for them: each cluster's rank-0 CTA takes the next ticket from a global
// counter when it starts an item (its first ticket is the cluster index) and
// publishes the item to every CTA of the cluster.  Tickets 0 .. NB - 1 are
// whole 32-token blocks; tickets NB .. NB + k R - 1 are column parts
// ("units") of the R last blocks, a block's k parts on consecutive tickets:
// unit v = r k + p is part p of block NB + r and covers column groups
// [p G / k, (p + 1) G / k) (a group is the KCL adjacent 64-column chunks the
// CTAs of a cluster take at once).  A cluster that finishes early simply takes
// more tickets, so clusters that run slower (by placement) do not set the
// kernel's time, and the last blocks are cut so the final ones end together
// ("[FlyDSL] Single-launch Mega-mHC on gfx950", Kernel Architecture: the
// split-K fallback at the wave edge).  The units of a block are summed
// through the global workspace; a cluster keeps its units' x in tensor memory
// and normalises them after its last item, once every part of their block is
// in, and it stops taking tickets before its tensor memory is full (the
// clusters together hold every unit, so the waits always end).

// Global workspace of the schedule and the split blocks: the ticket counter
// and the count of clusters that stopped taking tickets, then per split block
// r a row of counters (s_x arrivals, s_x reads, one owner-arrival count per CTA
// rank), then per unit the s_x partials of each CTA and the owner CTAs' summed
// projections.
constexpr int kMaxSplitBlocks = 64;
constexpr int kMaxUnits = 128;
constexpr int kCntStride = 32;
constexpr int kSchedRow = kMaxSplitBlocks;  // counter row of the ticket counter (word 0) and stop count (word 1)
constexpr size_t kSplitCntBytes = (size_t)(kMaxSplitBlocks + 1) * kCntStride * 4;
constexpr size_t kSplitSxFloats = (size_t)kMaxUnits * 16 * 32;  // [unit][rank][token]
constexpr size_t kSplitPpFloats = (size_t)kMaxUnits * 32 * 32;  // [unit][rank * slots + slot][part]

struct SplitWs {
  unsigned* cnt;
  float* sxp;
  float* pp;
  __device__ __forceinline__ SplitWs(char* w)
      : cnt(reinterpret_cast<unsigned*>(w)),
        sxp(reinterpret_cast<float*>(w + kSplitCntBytes)),
        pp(reinterpret_cast<float*>(w + kSplitCntBytes) + kSplitSxFloats) {}
};

// Bounded wait for a global counter to reach `target` (acquire); the same
// two tiers as the barrier waits.
__device__ __forceinline__ bool wait_count(const Ctx& x, const unsigned* p, unsigned target) {
  uint64_t t0 = 0;
  while (ld_acquire_gpu(p) < target) {
    if (wait_gave_up(x, t0)) return false;
    __nanosleep(100);
  }
  return true;
}

// s_x of a split block, summed over every CTA of every part of the block in a
// fixed order (the same value everywhere), after a bounded wait until all of
// them are in; the last of the block's readers resets its counters for the
// next call.  The loads go out in groups of eight, so their latencies
// overlap.  Out of line: only units take it.  Returns (the sum, 1), or
// (0, 0) when the call was abandoned.
__device__ __noinline__ float2 unit_sx(const Ctx x, const SplitWs w, int r, int k, int kcl, int lane) {
  const unsigned target = (unsigned)(k * kcl);
  if (!__all_sync(0xffffffffu, wait_count(x, &w.cnt[r * kCntStride], target))) return make_float2(0.f, 0.f);
  const int n = k * kcl;
  const float* base = w.sxp + (size_t)r * k * kcl * 32 + lane;  // units r k .. r k + k - 1 are adjacent
  float sx = 0.f;
  for (int e0 = 0; e0 < n; e0 += 8) {
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = e0 + q < n ? __ldcg(base + (size_t)(e0 + q) * 32) : 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) sx += v[q];
  }
  __syncwarp();
  if (lane == 0) {
    const unsigned old = atomicAdd(&w.cnt[r * kCntStride + 1], 1u);
    if (old == target * 8 - 1) {
      w.cnt[r * kCntStride] = 0;
      w.cnt[r * kCntStride + 1] = 0;
    }
  }
  return make_float2(sx, 1.f);
}

}  // namespace

// Owner side of a unit (exchange warp, out of line: only units take it).  The
// owner CTA publishes its tokens' cluster-summed projections and s_R of the
// unit; the owner that completes the k parts of the block last for its rank
// adds them in part order (the result does not depend on who is last) and
// finishes its tokens' gates.  pbuf holds the unit's sums on entry.
static __device__ __noinline__ void unit_owner_finish(const SeamArgs& a, unsigned* cnt, float* pp, float (*pbuf)[26],
                                               const float* ab, int r, int v, int k, int rank, int kcl, int slots,
                                               int64_t tok0, int lane) {
  constexpr int kParts = 25;
  for (int e = lane; e < slots * kParts; e += 32) {
    const int sl = e / kParts, q = e - sl * kParts;
    pp[((size_t)v * 32 + rank * slots + sl) * 32 + q] = pbuf[sl][q];
  }
  __threadfence();
  __syncwarp();
  unsigned old = 0;
  if (lane == 0) old = atom_add_acq_rel_gpu(&cnt[r * 32 + 2 + rank], 1u);
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != (unsigned)k - 1) return;
  (void)ld_acquire_gpu(&cnt[r * 32 + 2 + rank]);
  for (int e = lane; e < slots * kParts; e += 32) {
    const int sl = e / kParts, q = e - sl * kParts;
    const float* src = pp + ((size_t)r * k * 32 + rank * slots + sl) * 32 + q;  // part p of block r: unit r k + p
    float s = 0.f;
    for (int p0 = 0; p0 < k; p0 += 8) {
      float vv[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) vv[t] = p0 + t < k ? __ldcg(src + (size_t)(p0 + t) * 32 * 32) : 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) s += vv[t];
    }
    pbuf[sl][q] = s;
  }
  __syncwarp();
  if (lane < slots) {
    const int64_t tt = tok0 + rank + kcl * lane;
    if (tt < a.T) finish_store_gates(a, tt, &pbuf[lane][0], ab, a.H);
  }
  __syncwarp();
  if (lane == 0) cnt[r * 32 + 2 + rank] = 0;  // every part has arrived: reset for the next call
}

// FORM: 0 no_post (R' = comb . R), 1 post (+ post (x) Y), 2 identity: the
// first block's form, R' = R, no residual write.
// OUT: 0 bf16 norm, 1 mxfp8 (+ e4m3 codes, e8m0 scales), 2 fp8_grid (+ the
// quantisation dequantised to bf16)
// SCHED: how the clusters get their items.  0: blocks cid, cid + ncl, ...
// (static); 1: tickets from a global counter (a cluster that runs slower
// takes fewer blocks); 2: tickets, and the blocks of the partial last round
// cut into column parts (units).  The ticket ring and the unit paths are
// compiled only where used: the kernel's instruction footprint sets how well
// its hot loops stay in the instruction cache (measured: 2 to 25 % of the
// streaming time, by form).
template <int FORM, int OUT, bool MS, int KCL, int SCHED>
__global__ void __launch_bounds__(threads_of<OUT>(), 1)
    stream_seam_kernel(const __grid_constant__ SeamArgs a, const __grid_constant__ CUtensorMap tmR,
                       const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmRo,
                       const __grid_constant__ CUtensorMap tmFn, const __grid_constant__ CUtensorMap tmN,
                       const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmGc,
                       const __grid_constant__ CUtensorMap tmGp, const __grid_constant__ CUtensorMap tmGq,
                       int block0, int NB, int R, int k_parts, int G_groups, char* wsx,
                       unsigned long long report_ns, unsigned long long abort_ns) {
  constexpr bool DYN = SCHED >= 1, SPLIT = SCHED == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr bool LEAN = FORM == 2 && !MS;  // the MMAs read R' = R from the input stage
  using G = Geo<KCL, OUT, LEAN>;
  constexpr uint32_t kOutStage = G::kOutStage;
  constexpr uint32_t kOffNormT = G::kOffNormT, kOffCodesT = G::kOffCodesT, kPassCodes = G::kPassCodes;
  constexpr int kThreads = threads_of<OUT>();
  constexpr bool POST = FORM == 1, IDENT = FORM == 2;
  constexpr int kNI = LEAN ? G::kNILean : in_stages<FORM, KCL>();
  constexpr uint32_t kInStageF = in_stage_bytes<FORM>();
  static_assert(kNI <= kNIMax && kNI * kInStageF <= G::kInRing, "input ring");
  constexpr int kCl = G::kCl, kSlots = G::kSlots;
  constexpr uint32_t kOffIn = G::kOffIn, kXsBytes = G::kXsBytes, kRecvBytes = G::kRecvBytes;
  // readers of each published item in a CTA: input producer, fn producer, MMA
  // issuer (tcgen05 form), eight compute warps, store warp, grid warps, exchange warp
  constexpr int kReaders = 1 + 1 + (MS ? 0 : 1) + 8 + 1 + (OUT == 2 ? 3 : 0) + 1;
  typename G::Tail* tl = reinterpret_cast<typename G::Tail*>(sm + G::kOffTail);
  const Ctx X{&a, &tl->reported, &tl->aborted, report_ns, abort_ns};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int H = a.H;
  const int64_t T = a.T;
  // CTA r owns the 64-column chunks r, r + KCL, r + 2 KCL, ... of H (group g
  // holds chunks g KCL .. g KCL + KCL - 1): at any time the CTAs of a cluster
  // touch adjacent 128-byte pieces of the same rows
  const int n64 = H / kChunk;
  const int nch = n64 > (int)rank ? (n64 - (int)rank + kCl - 1) / kCl : 0;
  const int cid = blockIdx.x / kCl, ncl = gridDim.x / kCl;
  const SplitWs W(wsx);
  // chunks of this CTA in an item (a unit covers whole groups only)
  auto nchi = [&](const Item& it) { return SPLIT && it.unit >= 0 ? it.ng : nch; };

  // ---- the item list.  Static (SCHED 0): the cluster takes blocks cid,
  // cid + ncl, cid + 2 ncl, ... (every item a whole block, known to every
  // role without any exchange).  With tickets, rank 0 takes them from a
  // global counter and publishes each item to its cluster: item i sits in
  // slot i % kSchedD of each CTA's ring from its arrival until every reader
  // released it (at the end of its work on the item); its fields are read
  // from there where they are used, so no register holds them across the
  // chunk loops.
  volatile Item* const ring = tl->sched;
  auto iblock = [&](int i) -> int {
    return DYN ? ring[i % kSchedD].block : cid + i * ncl < NB ? block0 + cid + i * ncl : -1;
  };
  auto ig0 = [&](int i) -> int { return SPLIT ? ring[i % kSchedD].g0 : 0; };
  auto iunit = [&](int i) -> int { return SPLIT ? ring[i % kSchedD].unit : -1; };
  auto inch = [&](int i) -> int { return SPLIT && ring[i % kSchedD].unit >= 0 ? ring[i % kSchedD].ng : nch; };
  auto item = [&](int i) -> Item {
    return DYN ? const_cast<const Item&>(ring[i % kSchedD]) : Item{iblock(i), 0, G_groups, -1};
  };
  auto arrived = [&](int i) -> bool { return !DYN || wait_local(X, &tl->sched_full[i % kSchedD], (i / kSchedD) & 1); };
  auto arrived_warp = [&](int i) -> bool {
    return !DYN || wait_warp(X, &tl->sched_full[i % kSchedD], (i / kSchedD) & 1);
  };
  // one thread per reader role: the slot may be reused once every reader of
  // the cluster released it (a remote arrive on rank 0's sched_free).  The
  // arrive is relaxed: every read of the slot has returned before it (the
  // values decided the branches that lead here), and a release at cluster
  // scope was measured to stall the compute warps 2.5 us per item.
  auto release = [&](int i) {
    if (DYN) mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&tl->sched_free[i % kSchedD]), 0));
  };

  if (tid == 0) {
    for (int s = 0; s < kNI; ++s) {
      mbar_init(&tl->in_full[s], 1);
      mbar_init(&tl->in_empty[s], LEAN ? 9 : 8);  // (LEAN: and the MMAs that read the stage)
    }
    for (int s = 0; s < kNF; ++s) {
      mbar_init(&tl->fn_full[s], 1);
      mbar_init(&tl->fn_empty[s], MS ? 8 : 1);
    }
    for (int s = 0; s < kNO; ++s) {
      mbar_init(&tl->out_full[s], 8);
      // released by the store warp, and the MMA commit (the warp-level MMA warps)
      // unless the MMAs read the input stage, and the grid warp
      mbar_init(&tl->out_empty[s], (MS ? 9 : LEAN ? 1 : 2) + (OUT == 2 ? 1 : 0));
    }
    mbar_init(&tl->d_full, 1);
    for (int p = 0; p < 2; ++p) {
      mbar_init(&tl->gates_full[p], 1);
      mbar_init(&tl->gates_empty[p], 8);
    }
    mbar_init(&tl->dbuf_full, 4);  // the four D readers (or folders)
    mbar_init(&tl->dbuf_free, 1);  // the exchange warp
    mbar_init(&tl->d_free, 4);     // the four D readers
    mbar_init(&tl->mma_fin, 1);
    mbar_init(&tl->fold_full, 4);  // warps 4-7 (warp-MMA form)
    for (int p = 0; p < 2; ++p) {
      mbar_init(&tl->xs_full[p], 1);    // + kXsBytes of st.async from the cluster
      mbar_init(&tl->recv_full[p], 1);  // + kRecvBytes of st.async from the cluster
      mbar_init(&tl->recv_free[p], kCl);
      mbar_init(&tl->red_full[p], 8);
      mbar_init(&tl->red_free[p], 1);   // the exchange warp has read the partials
    }
    for (int s = 0; s < kSchedD; ++s) {
      mbar_init(&tl->sched_full[s], 1);               // + 16 bytes of st.async from rank 0
      mbar_init(&tl->sched_free[s], kCl * kReaders);  // (rank 0) every reader of the cluster
    }
    tl->reported = 0;
    tl->aborted = 0;
    tl->nunits = 0;
    mbar_fence_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tmR);
    if (POST) prefetch_tmap(&tmY);
    if (!IDENT) prefetch_tmap(&tmGc);
    prefetch_tmap(&tmGp);
    if (POST) prefetch_tmap(&tmGq);
  }
  if (warp == 10 && lane == 0) prefetch_tmap(&tmFn);
  if (warp == 12 && lane == 0) {
    if (!IDENT) prefetch_tmap(&tmRo);
    prefetch_tmap(&tmN);
    if (OUT == 1) prefetch_tmap(&tmC);
  }
  if (warp == 9) {
    tmem_alloc(&tl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // barriers initialised in every CTA of the cluster
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  // Programmatic dependent launch: everything above (barriers, tensor memory,
  // the cluster barrier, tensor-map prefetch) may overlap the previous kernel
  // on the stream; every read of global memory comes after this wait, which
  // returns once that kernel has completed and its writes are visible.  The
  // next kernel may then begin its own set-up while this one runs.
  griddep_wait();
  if (tid == 0) griddep_launch_dependents();
  // gamma of this CTA's first chunks (groups), staged once by the compute
  // warps, its only readers (the producers start loading meanwhile)
  if (warp < 8) {
    for (int i = tid; i < min(nch, G::kGamChunks) * 8; i += 256)
      tl->gam[i >> 3][i & 7] = __ldg(reinterpret_cast<const uint4*>(a.gamma + ((i >> 3) * kCl + (int)rank) * kChunk) + (i & 7));
    named_bar_sync(1, 256);
  }

  if (warp == 8) {
    // --------------------------------------------------- input producer --
    if (lane == 0) {
      // evict-normal, not evict-first: measured 5 % faster (the neighbouring
      // CTAs of the cluster read the other halves of the promoted 256-byte
      // L2 lines at about the same time)
      const uint64_t pol = l2_evict_normal();
      const uint32_t bytes = (POST ? 5 : 4) * kRTile;
      // Rank 0 publishes the cluster's items, one ahead of its own loads: the
      // next ticket, decoded, to every CTA of the cluster.
      const int cap = MS ? kMaxChunks : kMaxChunksTC;  // tensor-memory x slots a cluster's units may fill
      const int maxng = k_parts > 1 ? (G_groups + k_parts - 1) / k_parts : 0;
      int pub = 0, used = 0, nunits = 0;
      bool ended = false;
      auto publish = [&]() -> bool {
        const int s = pub % kSchedD;
        // every reader of the item kSchedD before has read its slot
        if (!wait_local(X, &tl->sched_free[s], ((pub / kSchedD) & 1) ^ 1)) return false;
        Item it{-1, 0, 0, -1};
        if (!ended) {
          int t = 0x7fffffff;
          if (pub == 0) {
            t = cid;
          } else if (!SPLIT || (used + maxng <= cap && nunits < kMaxUnitsCl)) {
            t = (int)atomicAdd(&W.cnt[kSchedRow * kCntStride], 1u) + ncl;
          }
          if (t < NB) {
            it = Item{block0 + t, 0, G_groups, -1};
          } else if (SPLIT && t < NB + k_parts * R) {
            const int v = t - NB, r = v / k_parts, p = v - r * k_parts;
            const int g0 = p * G_groups / k_parts, g1 = (p + 1) * G_groups / k_parts;
            it = Item{block0 + NB + r, g0, g1 - g0, v};
            used += g1 - g0;
            ++nunits;
          } else {
            ended = true;
            // the last cluster to stop taking tickets resets the counters for the next call
            if (atomicAdd(&W.cnt[kSchedRow * kCntStride + 1], 1u) == (unsigned)ncl - 1) {
              W.cnt[kSchedRow * kCntStride] = 0;
              W.cnt[kSchedRow * kCntStride + 1] = 0;
            }
          }
        }
        const uint32_t da = smem_u32(&tl->sched[s]), db = smem_u32(&tl->sched_full[s]);
        for (int dst = 0; dst < kCl; ++dst)
          st_async_v4(mapa_shared(da, (uint32_t)dst), it.block, it.g0, it.ng, it.unit, mapa_shared(db, (uint32_t)dst));
        ++pub;
        return true;
      };
      int j = 0, ng = 0;  // input-stage loads and gate loads issued
      // Item n's phase of its ring slot (armed by this CTA, completed by rank
      // 0's 16 bytes), then, for a real item, its carried gates into buffer
      // n % 2 once item n - 2 has finished with that buffer.  The gates are
      // fetched an item ahead (during item n - 1, once its compute has begun),
      // so their load latency never stalls the compute warps between items.
      auto next_item = [&](int n) -> bool {
        if (DYN) mbar_arrive_expect_tx(&tl->sched_full[n % kSchedD], (uint32_t)sizeof(Item));
        if (!arrived(n)) return false;
        const int b = iblock(n);
        if (b < 0) return true;
        const int gbuf = n & 1, tn = b * kBM;
        if (!wait_local(X, &tl->gates_empty[gbuf], ((n >> 1) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(&tl->gates_full[gbuf], (IDENT ? 4 : POST ? 24 : 20) * kBM * 4);
        if (!IDENT) tma_load_2d(&tl->gates[gbuf].comb[0][0], &tmGc, &tl->gates_full[gbuf], 0, tn, pol);
        tma_load_2d(&tl->gates[gbuf].pre[0][0], &tmGp, &tl->gates_full[gbuf], 0, tn, pol);
        if (POST) tma_load_2d(&tl->gates[gbuf].post[0][0], &tmGq, &tl->gates_full[gbuf], 0, tn, pol);
        ++ng;
        return true;
      };
      // Item i's loads; at its first step rank 0 publishes item i + 1, and
      // once this item's compute has begun (its load for chunk kNI waited for
      // chunk 0 to be consumed), or at its last step, item i + 1's gates are
      // fetched.  Item -1 has no chunks: it publishes and fetches item 0.
      // (One call site each keeps the producer's code small.)
      bool ok = true;
      for (int i = -1; ok; ++i) {
        int t0 = 0, gb = 0, ni = 0;
        if (i >= 0) {
          const Item it = item(i);
          if (it.block < 0) {
            release(i);
            break;
          }
          if (SPLIT && it.unit >= 0) {  // the cluster's units, for the normalise-only passes after its last item
            tl->ulist[tl->nunits] = it;
            ++tl->nunits;
          }
          t0 = it.block * kBM;
          gb = it.g0;
          ni = nchi(it);
        }
        const int steps = ni > 0 ? ni : 1, cg = ni - 1 < kNI ? steps - 1 : kNI;
        for (int c = 0; c < steps; ++c) {
          if (c < ni) {
            const int s = j % kNI;
            if (!(ok = wait_local(X, &tl->in_empty[s], ((j / kNI) & 1) ^ 1))) break;
            uint8_t* st = sm + kOffIn + s * kInStageF;
            const int h = ((gb + c) * kCl + (int)rank) * kChunk;
            mbar_arrive_expect_tx(&tl->in_full[s], bytes);
            // the four streams' tiles in one copy: box [64 columns, 32 tokens, 4 streams]
            tma_load_3d(st, &tmR, &tl->in_full[s], h, t0, 0, pol);
            if (POST) tma_load_2d(st + 4 * kRTile, &tmY, &tl->in_full[s], h, t0, pol);
            ++j;
          }
          if (DYN && c == 0 && rank == 0 && !(ok = publish())) break;
          if (c == cg && !(ok = next_item(i + 1))) break;
        }
        if (ok && i >= 0) release(i);
      }
      // Every load issued lands before the CTA exits.  A stage is refilled
      // only after all eight compute warps released it, and they release it
      // only after seeing its previous load complete, so only the last load
      // of each stage (and of each gate buffer) can still be in flight.
      for (int jj = (j > kNI ? j - kNI : 0); jj < j; ++jj) drain(X, &tl->in_full[jj % kNI], (jj / kNI) & 1);
      for (int q = (ng > 2 ? ng - 2 : 0); q < ng; ++q) drain(X, &tl->gates_full[q & 1], (q >> 1) & 1);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------ fn producer --
    if (lane == 0) {
      const uint64_t pol = l2_evict_last();
      int j = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        if (!(ok = arrived(i))) break;
        if (iblock(i) < 0) {
          release(i);
          break;
        }
        const int gb = ig0(i), ni = inch(i);
        for (int c = 0; c < ni; ++c, ++j) {
          const int f = j % kNF;
          if (!(ok = wait_local(X, &tl->fn_empty[f], ((j / kNF) & 1) ^ 1))) break;
          uint8_t* st = sm + kOffFn + f * kFnStage;
          const int h = ((gb + c) * kCl + (int)rank) * kChunk;
          mbar_arrive_expect_tx(&tl->fn_full[f], kFnStage);
          // the four streams' fn tiles in one copy: box [64 columns, 48 rows, 4 streams]
          tma_load_3d(st, &tmFn, &tl->fn_full[f], h, 0, 0, pol);
        }
        if (ok) release(i);
      }
      // as for the input ring: only the last load of each fn stage can still be in flight
      for (int jj = (j > kNF ? j - kNF : 0); jj < j; ++jj) drain(X, &tl->fn_full[jj % kNF], (jj / kNF) & 1);
    }
  } else if (warp == 9) {
    // -------------------------------------- tcgen05 projection (one thread) --
    if (!MS && lane == 0) {
      int j = 0, jr = 0, nu = 0;
      bool ok = arrived(0);
      for (int i = 0; ok && iblock(i) >= 0; ++i) {
        const int ni = inch(i);
        for (int c = 0; c < ni; ++c, ++j) {
          const int o = j % kNO;
          const int f = jr % kNF, si = jr % kNI;  // (LEAN: chunk jr's input stage)
          // the chunk's R': in the compute warps' output stage, or (LEAN) the
          // input stage itself as soon as its load has landed
          if (!(ok = LEAN ? wait_local(X, &tl->in_full[si], (jr / kNI) & 1)
                          : wait_local(X, &tl->out_full[o], (j / kNO) & 1)))
            break;
          // the first MMA of an item overwrites D: the previous item's D must have been read
          if (c == 0 && i > 0 && !(ok = wait_local(X, &tl->d_free, (i - 1) & 1))) break;
          if (!(ok = wait_local(X, &tl->fn_full[f], (jr / kNF) & 1))) break;
          tc_fence_after();
          // R' of the 4 streams [128 x 64], fn of the 4 streams [192 x 64]
          const uint32_t ra = smem_u32(LEAN ? sm + kOffIn + si * kInStageF : sm + kOffOut + o * kOutStage);
          const uint32_t fb = smem_u32(sm + kOffFn + f * kFnStage);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tmem + kColD, sdesc_k_sw128(ra + kk * 32), sdesc_k_sw128(fb + kk * 32), kIdesc, (c | kk) != 0);
          tc_commit(&tl->fn_empty[f]);
          tc_commit(LEAN ? &tl->in_empty[si] : &tl->out_empty[o]);
          if (c == ni - 1) tc_commit(&tl->d_full);
          ++jr;
        }
        if (!ok) break;
        const bool full = iunit(i) < 0;
        if (!full) ++nu;
        if (!(ok = arrived(i + 1))) break;
        const int nblk = iblock(i + 1);
        // normalise-only passes after this item (of this item when the next
        // covers other columns or there is none; of every unit after the
        // last): one stage per group of chunks, no MMA
        // (LEAN: the MMAs never hold an output stage)
        const int qa = full ? -1 : 0, qb = LEAN ? -1 : full ? (nblk < 0 || iunit(i + 1) >= 0 ? 0 : -1) : (nblk < 0 ? nu : 0);
        for (int q = qa; q < qb && ok; ++q) {
          const int nq = !SPLIT || q < 0 ? nch : const_cast<const Item&>(tl->ulist[q]).ng;
          for (int c0 = 0; c0 < nq; c0 += G::kNormGroup, ++j) {
            if (!(ok = wait_local(X, &tl->out_full[j % kNO], (j / kNO) & 1))) break;
            mbar_arrive(&tl->out_empty[j % kNO]);
          }
        }
        release(i);
        if (ok && nblk < 0) release(i + 1);  // the end of the list
      }
      // every MMA issued (and the commits before it) completes before the CTA
      // exits and tensor memory is freed
      tc_commit(&tl->mma_fin);
      drain(X, &tl->mma_fin, 0);
    }
  } else if (warp == 12) {
    // ---------------------------- stores: R' tiles, norm tile, e4m3 codes --
    // (no norm pointer: the first pass of the unshifted ordering, which keeps
    // R' and the gates only)
    const bool store_norm = a.norm != nullptr;
    int j = 0, nu = 0;
    // lane = token: the ue8m0 codes of one norm tile (two 32-column groups)
    auto quant_tile = [&](const uint8_t* nt, uint8_t* ct, int64_t tp, int h) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t nb[16];
#pragma unroll
        for (int jq = 0; jq < 4; ++jq) {
          const int ch = 4 * half + jq;
          uint4 v = *reinterpret_cast<const uint4*>(nt + lane * 128 + ((ch ^ (lane & 7)) << 4));
          nb[4 * jq] = v.x; nb[4 * jq + 1] = v.y; nb[4 * jq + 2] = v.z; nb[4 * jq + 3] = v.w;
        }
        uint32_t cw[8];
        const uint8_t sb = quant_group32(nb, cw, a.amax_floor);
        uint4* cd = reinterpret_cast<uint4*>(ct + lane * 64 + 32 * half);
        cd[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        cd[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        const int64_t tt = tp + lane;
        if (tt < T) a.scales[tt * (H / 32) + (h + 32 * half) / 32] = sb;
      }
    };
    // (lane 0) a stage is given back once the bulk stores issued from it have
    // read it.  With the fp8_grid output, and in the identity form whose
    // stages hold only the norm tile, the newest group may still be reading:
    // its stage is given back after the next group is committed (the compute
    // warps need it only kNO - 1 stages later), so the store warp never waits
    // on its own stores; measured: fp8_grid at T = 16384 396 to 386 us, the
    // identity form 193 to 191 us, but 3 to 4 us slower for the bf16 post and
    // no_post forms, whose stages turn over faster.
    int pend = -1;
    auto retire = [&](int o) {
      tma_store_commit();
      if (OUT == 2 || LEAN) {
        tma_store_wait_read_1();  // every group but the newest has read its stage
        if (pend >= 0) mbar_arrive(&tl->out_empty[pend]);
        pend = o;
      } else {
        tma_store_wait_read_all();
        mbar_arrive(&tl->out_empty[o]);
      }
    };
    int prevblk = -1;  // the previous item's block when it was a whole block, else -1
    bool ok = arrived_warp(0);
    for (int i = 0; ok && iblock(i) >= 0; ++i) {
      // this item's chunks carry the previous item's norm when both are whole blocks
      const bool full = iunit(i) < 0, fused = prevblk >= 0 && full;
      const int t0 = iblock(i) * kBM, tp = fused ? prevblk * kBM : 0, gb = ig0(i), ni = inch(i);
      for (int c = 0; c < ni; ++c, ++j) {
        const int o = j % kNO;
        uint8_t* ost = sm + kOffOut + o * kOutStage;
        const int h = ((gb + c) * kCl + (int)rank) * kChunk;
        if (!(ok = wait_warp(X, &tl->out_full[o], (j / kNO) & 1))) break;
        if (OUT == 1 && fused) {
          quant_tile(ost + kOffNormT, ost + kOffCodesT, tp, h);
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          if (!IDENT) {
            tma_store_3d(&tmRo, ost, h, t0, 0);  // the four R' tiles in one copy
          }
          if (fused) {
            if (store_norm) tma_store_2d(&tmN, ost + kOffNormT, h, tp);
            if (OUT == 1) tma_store_2d(&tmC, ost + kOffCodesT, h, tp);
          }
          retire(o);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (!full) ++nu;
      if (!(ok = arrived_warp(i + 1))) break;
      const int nblk = iblock(i + 1);
      // normalise-only passes: the norm tiles of a group of chunks per stage
      const int qa = full ? -1 : 0, qb = full ? (nblk < 0 || iunit(i + 1) >= 0 ? 0 : -1) : (nblk < 0 ? nu : 0);
      constexpr int NG = G::kNormGroup;
      for (int q = qa; q < qb && ok; ++q) {
        const Item u = !SPLIT || q < 0 ? item(i) : const_cast<const Item&>(tl->ulist[q]);
        const int tq = u.block * kBM, gq = u.g0, nq = nchi(u);
        for (int c0 = 0; c0 < nq; c0 += NG, ++j) {
          const int o = j % kNO;
          uint8_t* ost = sm + kOffOut + o * kOutStage;
          if (!(ok = wait_warp(X, &tl->out_full[o], (j / kNO) & 1))) break;
          const int ng = min(NG, nq - c0);
          if (OUT == 1) {  // codes tiles in stage slot 4
            for (int g = 0; g < ng; ++g)
              quant_tile(ost + g * kRTile, ost + kPassCodes + g * 2048, tq, ((gq + c0 + g) * kCl + (int)rank) * kChunk);
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (lane == 0) {
            for (int g = 0; g < ng; ++g) {
              const int h = ((gq + c0 + g) * kCl + (int)rank) * kChunk;
              if (store_norm) tma_store_2d(&tmN, ost + g * kRTile, h, tq);
              if (OUT == 1) tma_store_2d(&tmC, ost + kPassCodes + g * 2048, h, tq);
            }
            retire(o);
          }
          __syncwarp();
        }
      }
      prevblk = full ? iblock(i) : -1;
      __syncwarp();
      if (lane == 0) {
        release(i);
        if (ok && nblk < 0) release(i + 1);  // the end of the list
      }
    }
    // every bulk store issued has read its shared memory and written global
    // memory before the CTA exits (the hardware wait always ends); the last
    // stage is given back too
    if (lane == 0) {
      tma_store_wait_all();
      if (pend >= 0) mbar_arrive(&tl->out_empty[pend]);
    }
  } else if (OUT == 2 && warp >= 13) {
    // ------------------------------------------------------ grid warps --
    // fp8_grid: warp 13 + o reads the norm tiles of output stage o and writes
    // their grid (bf16 of the dequantised e4m3 codes) straight to global
    // memory; the stage is free again once it has read them.
    const int me = warp - 13;
    // the grid row of token tp + lane, columns h .. h + 63, from norm tile nt;
    // `rel` is released once the tile is read (the row is then in registers)
    auto grid_row = [&](const uint8_t* nt, uint64_t* rel, int64_t tp, int h) {
      const int64_t tt = tp + lane;
      grid_tile_row(nt, rel, tt < T ? a.grid + tt * H + h : nullptr, a.amax_floor, lane);
    };
    int j = 0, nu = 0, prevblk = -1;
    bool ok = arrived_warp(0);
    for (int i = 0; ok && iblock(i) >= 0; ++i) {
      const bool full = iunit(i) < 0, fused = prevblk >= 0 && full;
      const int64_t tp = fused ? (int64_t)prevblk * kBM : 0;
      const int gb = ig0(i), ni = inch(i);
      for (int c = 0; c < ni; ++c, ++j) {
        const int o = j % kNO;
        if (o != me) continue;
        const uint8_t* ost = sm + kOffOut + o * kOutStage;
        if (!(ok = wait_warp(X, &tl->out_full[o], (j / kNO) & 1))) break;
        if (fused) {
          grid_row(ost + kOffNormT, &tl->out_empty[o], tp, ((gb + c) * kCl + (int)rank) * kChunk);
        } else if (lane == 0) {
          mbar_arrive(&tl->out_empty[o]);
        }
      }
      if (!ok) break;
      if (!full) ++nu;
      if (!(ok = arrived_warp(i + 1))) break;
      const int nblk = iblock(i + 1);
      // normalise-only passes: the norm tiles of a group of chunks per stage
      const int qa = full ? -1 : 0, qb = full ? (nblk < 0 || iunit(i + 1) >= 0 ? 0 : -1) : (nblk < 0 ? nu : 0);
      constexpr int NG = G::kNormGroup;
      for (int q = qa; q < qb && ok; ++q) {
        const Item u = !SPLIT || q < 0 ? item(i) : const_cast<const Item&>(tl->ulist[q]);
        const int64_t tq = (int64_t)u.block * kBM;
        const int gq = u.g0, nq = nchi(u);
        for (int c0 = 0; c0 < nq; c0 += NG, ++j) {
          const int o = j % kNO;
          if (o != me) continue;
          const uint8_t* ost = sm + kOffOut + o * kOutStage;
          if (!(ok = wait_warp(X, &tl->out_full[o], (j / kNO) & 1))) break;
          const int ng = min(NG, nq - c0);
          for (int g = 0; g < ng; ++g)
            grid_row(ost + g * kRTile, g == ng - 1 ? &tl->out_empty[o] : nullptr, tq, ((gq + c0 + g) * kCl + (int)rank) * kChunk);
        }
      }
      prevblk = full ? iblock(i) : -1;
      __syncwarp();
      if (lane == 0) {
        release(i);
        if (ok && nblk < 0) release(i + 1);  // the end of the list
      }
    }
  } else if (warp == 11) {
    // ------------------------------------ exchange and gate finish warp --
    // Per item: (1) this CTA's s_x partials to every CTA of the cluster (each
    // forms rstd_x itself), (2) the 24 projections and s_R of each token to
    // its owner CTA (token % KCL), (3) the gates of the tokens this CTA owns.
    // Sends are st.async completing bytes on the receiver's mbarrier; the
    // compute warps only hand their partials over and go on.  recv_free keeps
    // the partials of item i + 2 out of a slot until every owner has read
    // item i from it.  A unit (a column part of a block) publishes its s_x
    // partials and its owners' sums in the global workspace instead of the
    // s_x exchange; the owner that completes a block's parts last finishes
    // its tokens' gates.
    if (lane < 27) tl->ab[lane] = lane < 3 ? a.alpha[lane] : a.bias[lane - 3];
    __syncwarp();
    for (int i = 0; arrived_warp(i) && iblock(i) >= 0; ++i) {
      const int b = iblock(i), par = i & 1, v = iunit(i);
      const bool unit = SPLIT && v >= 0;
      if (!wait_warp(X, &tl->red_full[par], (i >> 1) & 1)) break;
      float sx = 0.f, sR = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float2 v = tl->red[par][w][lane];
        sR += v.x;
        sx += v.y;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->red_free[par]);  // the compute warps may write item i + 2's partials
      if (unit) {  // this CTA's s_x partials of the unit, for every part's rstd_x
        W.sxp[((size_t)v * kCl + (int)rank) * 32 + lane] = sx;
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(&W.cnt[(v / k_parts) * kCntStride], 1u);
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&tl->xs_full[par], kXsBytes);
        const uint32_t xa = smem_u32(&tl->xs[par][rank][lane]), xb = smem_u32(&tl->xs_full[par]);
#pragma unroll
        for (int dst = 0; dst < kCl; ++dst)
          st_async_f32(mapa_shared(xa, (uint32_t)dst), sx, mapa_shared(xb, (uint32_t)dst));
      }
      if (!wait_warp(X, &tl->dbuf_full, i & 1)) break;
      if (i >= 2 && !wait_warp_remote(X, &tl->recv_free[par], ((i >> 1) & 1) ^ 1)) break;
      {
        const uint32_t dst = (uint32_t)(lane % kCl);
        const uint32_t ra = mapa_shared(smem_u32(&tl->recv[par][rank][lane / kCl][0]), dst);
        const uint32_t rb = mapa_shared(smem_u32(&tl->recv_full[par]), dst);
#pragma unroll 1
        for (int k = 0; k < 24; k += 2) {
          float s0 = tl->dbuf[0][lane][k], s1 = tl->dbuf[0][lane][k + 1];
#pragma unroll
          for (int q = 1; q < 4; ++q) {
            s0 += tl->dbuf[q][lane][k];
            s1 += tl->dbuf[q][lane][k + 1];
          }
          st_async_v2(ra + 4 * k, s0, s1, rb);
        }
        st_async_f32(ra + 4 * 24, sR, rb);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->dbuf_free);

      if (lane == 0) mbar_arrive_expect_tx(&tl->recv_full[par], kRecvBytes);
      if (!wait_warp(X, &tl->recv_full[par], (i >> 1) & 1)) break;
      // sums over the cluster, one (owned token, part) pair per lane and round
      for (int e = lane; e < kSlots * kOwnerParts; e += 32) {
        const int sl = e / kOwnerParts, k = e - sl * kOwnerParts;
        float s = 0.f;
#pragma unroll
        for (int src = 0; src < kCl; ++src) s += tl->recv[par][src][sl][k];
        tl->pbuf[sl][k] = s;
      }
      __syncwarp();
      if (lane < kCl) mbar_arrive_remote(mapa_shared(smem_u32(&tl->recv_free[par]), lane));
      if (!unit) {
        if (lane < kSlots) {
          const int64_t tt = (int64_t)b * kBM + (int)rank + kCl * lane;
          if (tt < T) finish_store_gates(a, tt, &tl->pbuf[lane][0], tl->ab, H);
        }
      } else {
        unit_owner_finish(a, W.cnt, W.pp, tl->pbuf, tl->ab, v / k_parts, v, k_parts, (int)rank, kCl, kSlots,
                          (int64_t)b * kBM, lane);
      }
      __syncwarp();
      if (lane == 0) release(i);
    }
  } else if (warp < 8) {
    // ---------------------------------------------------- compute warps --
    const int q4 = warp & 3, wq = warp >> 2;
    const uint32_t colx = MS ? 0u : kDCols;
    const uint32_t xaddr = tmem + ((uint32_t)(32 * q4) << 16) + colx + 8 * wq;
    const uint32_t off = lane * 128 + ((warp ^ (lane & 7)) << 4);  // row = token, 16-byte chunk = warp
    // gamma of the 8 columns of this warp in chunk c of group g
    auto gamma8 = [&](int g) -> uint4 {
      return g < G::kGamChunks ? tl->gam[g][warp]
                               : __ldg(reinterpret_cast<const uint4*>(a.gamma + (g * kCl + (int)rank) * kChunk + 8 * warp));
    };
    // Warp-level projection (MS): warp w owns stream w % 4 and the 32 columns
    // [32 (w / 4), +32) of every chunk: D[32 tokens x 24 logits] += R'[32 x 32]
    // . (fn_hi + fn_lo)[32 x 24], m16n8k16 MMAs with fp32 accumulation, one
    // chunk behind the R' writes of all eight warps.
    float acc[2][3][4];
    auto mma_chunk = [&](int jj, int jr) -> bool {
      const int oo = jj % kNO, ff = jr % kNF;
      if (!wait_warp(X, &tl->out_full[oo], (jj / kNO) & 1)) return false;
      if (!wait_warp(X, &tl->fn_full[ff], (jr / kNF) & 1)) return false;
      const uint32_t rt = smem_u32(sm + kOffOut + oo * kOutStage + (warp & 3) * kRTile);
      const uint32_t ft = smem_u32(sm + kOffFn + ff * kFnStage + (warp & 3) * kFnTile);
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int kg = 2 * (warp >> 2) + kk;  // 16-column group of the chunk
        uint32_t af[2][4], bq[3][4];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int row = 16 * m + (mi & 1) * 8 + rr, ch = 2 * kg + (mi >> 1);
          ldmatrix_x4(rt + row * 128 + ((ch ^ rr) << 4), af[m][0], af[m][1], af[m][2], af[m][3]);
        }
#pragma unroll
        for (int pq = 0; pq < 3; ++pq) {  // fn rows 16 pq .. 16 pq + 15 (n8 tiles 2 pq, 2 pq + 1)
          const int row = 16 * pq + (mi >> 1) * 8 + rr, ch = 2 * kg + (mi & 1);
          ldmatrix_x4(ft + row * 128 + ((ch ^ rr) << 4), bq[pq][0], bq[pq][1], bq[pq][2], bq[pq][3]);
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
          for (int n = 0; n < 3; ++n) {
            const int th = n, tlo = 3 + n;  // hi and lo rows of logits 8n .. 8n + 7
            mma_bf16_16816(acc[m][n], af[m][0], af[m][1], af[m][2], af[m][3], bq[th >> 1][2 * (th & 1)],
                           bq[th >> 1][2 * (th & 1) + 1]);
            mma_bf16_16816(acc[m][n], af[m][0], af[m][1], af[m][2], af[m][3], bq[tlo >> 1][2 * (tlo & 1)],
                           bq[tlo >> 1][2 * (tlo & 1) + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tl->out_empty[oo]);
        mbar_arrive(&tl->fn_empty[ff]);
      }
      return true;
    };

    float rprev = 0.f;
    // rstd_x of whole-block item fi (block b) from the s_x partials the CTAs of
    // the cluster sent (same sum order in every CTA, so all hold the same value)
    auto take_rstd = [&](int fi, int b) -> bool {
      const int pp = fi & 1;
      if (!wait_warp(X, &tl->xs_full[pp], (fi >> 1) & 1)) return false;
      float sx = 0.f;
#pragma unroll
      for (int src = 0; src < kCl; ++src) sx += tl->xs[pp][src][lane];
      const int64_t tt = (int64_t)b * kBM + lane;
      rprev = tt < T ? 1.0f / sqrtf(sx / (float)H + a.eps) : 0.f;
      return true;
    };

    // tcgen05 projection: warp q4 reads stream q4's diagonal block of item
    // ip's D (TMEM lanes 32 q4 .., columns 48 q4 .. 48 q4 + 47) during the
    // next item's first chunk, frees D for that item's MMAs, and hands the
    // hi + lo sums to the exchange warp through dbuf.
    auto read_d = [&](int ip, int nip) -> bool {
      float dv[48];
      if (nip > 0) {
        if (!wait_warp(X, &tl->d_full, ip & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 6; ++k)
          tc_ld_x8(tmem + ((uint32_t)(32 * warp) << 16) + kColD + 48 * warp + 8 * k, dv + 8 * k);
      } else {
#pragma unroll
        for (int k = 0; k < 48; ++k) dv[k] = 0.f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->d_free);
      if (!wait_warp(X, &tl->dbuf_free, (ip & 1) ^ 1)) return false;
      float* r0 = &tl->dbuf[warp][lane][0];
#pragma unroll
      for (int k = 0; k < 24; ++k) r0[k] = dv[k] + dv[24 + k];
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->dbuf_full);
      return true;
    };

    int j = 0, ji = 0, nu = 0, sbu = 0, nprev = 0;
    int prevblk = -1;  // the previous item's block when it was a whole block, else -1
    bool ok = arrived_warp(0);
    for (int i = 0; ok && iblock(i) >= 0; ++i) {
      // this item's chunks normalise the previous item's x (same columns)
      const bool full = iunit(i) < 0, fused = prevblk >= 0 && full;
      const int ni = inch(i), sb = full ? 0 : sbu;
      float2 comb2[16], post2[4], pre2[4];  // each gate duplicated for the fp32x2 FMAs
      {
        float4 gc[4], gp = make_float4(0.f, 0.f, 0.f, 0.f), gq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; ++k) gc[k] = gp;
        {  // rows past T arrive as zeros; the buffer is released at the item's end
          if (!(ok = wait_warp(X, &tl->gates_full[i & 1], (i >> 1) & 1))) break;
          const GateTile& gt = tl->gates[i & 1];
          if (!IDENT) {
#pragma unroll
            for (int k = 0; k < 4; ++k) gc[k] = *reinterpret_cast<const float4*>(&gt.comb[lane][4 * k]);
          }
          gp = *reinterpret_cast<const float4*>(&gt.pre[lane][0]);
          if (POST) gq = *reinterpret_cast<const float4*>(&gt.post[lane][0]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          comb2[4 * k] = make_float2(gc[k].x, gc[k].x); comb2[4 * k + 1] = make_float2(gc[k].y, gc[k].y);
          comb2[4 * k + 2] = make_float2(gc[k].z, gc[k].z); comb2[4 * k + 3] = make_float2(gc[k].w, gc[k].w);
        }
        pre2[0] = make_float2(gp.x, gp.x); pre2[1] = make_float2(gp.y, gp.y);
        pre2[2] = make_float2(gp.z, gp.z); pre2[3] = make_float2(gp.w, gp.w);
        post2[0] = make_float2(gq.x, gq.x); post2[1] = make_float2(gq.y, gq.y);
        post2[2] = make_float2(gq.z, gq.z); post2[3] = make_float2(gq.w, gq.w);
      }
      float2 sR2 = make_float2(0.f, 0.f), sx2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < 3; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[m][n][e] = 0.f;

      for (int c = 0; c < ni; ++c, ++j) {
        const int o = j % kNO;
        uint32_t ow[4][4];
        float x[8];
        // the previous item's x and gamma of these columns, fetched now so
        // their latency hides behind this chunk's post-mix
        uint32_t xr[8];
        uint4 gv = make_uint4(0, 0, 0, 0);
        if (fused) {  // (a whole block: its column groups start at 0)
          tc_ld_x8_issue(xaddr + 16 * c, xr);
          gv = gamma8(c);
        }
        {
          const int s = ji % kNI;
          if (!(ok = wait_warp(X, &tl->in_full[s], (ji / kNI) & 1))) break;
          const uint8_t* st = sm + kOffIn + s * kInStageF;
          uint4 rin[4], yin = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int q = 0; q < 4; ++q) rin[q] = *reinterpret_cast<const uint4*>(st + q * kRTile + off);
          if (POST) yin = *reinterpret_cast<const uint4*>(st + 4 * kRTile + off);
          __syncwarp();
          if (lane == 0) mbar_arrive(&tl->in_empty[s]);
          ++ji;
          // two columns at a time with packed fp32x2 FMAs (each half rounds like a scalar FMA)
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
            const float2 r0 = bf16pair((&rin[0].x)[wd]), r1 = bf16pair((&rin[1].x)[wd]);
            const float2 r2 = bf16pair((&rin[2].x)[wd]), r3 = bf16pair((&rin[3].x)[wd]);
            const float2 yy = bf16pair((&yin.x)[wd]);
            float2 xx = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w;
              if (IDENT) {
                w = (&rin[q].x)[wd];  // R' = R, bit for bit
              } else {
                float2 v = __fmul2_rn(comb2[4 * q], r0);
                v = __ffma2_rn(comb2[4 * q + 1], r1, v);
                v = __ffma2_rn(comb2[4 * q + 2], r2, v);
                v = __ffma2_rn(comb2[4 * q + 3], r3, v);
                if (POST) v = __ffma2_rn(post2[q], yy, v);
                w = pack_bf16x2(v.x, v.y);
              }
              ow[q][wd] = w;
              const float2 rr2 = bf16pair(w);
              sR2 = __ffma2_rn(rr2, rr2, sR2);
              xx = __ffma2_rn(pre2[q], rr2, xx);
            }
            x[2 * wd] = xx.x;
            x[2 * wd + 1] = xx.y;
            sx2 = __ffma2_rn(xx, xx, sx2);
          }
        }
        if (fused && c == 0 && !(ok = take_rstd(i - 1, prevblk))) break;
        if (!(ok = wait_warp(X, &tl->out_empty[o], ((j / kNO) & 1) ^ 1))) break;
        uint8_t* ost = sm + kOffOut + o * kOutStage;
        if (!LEAN) {  // (LEAN: the MMAs read R' = R from the input stage)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(ost + q * kRTile + off) = make_uint4(ow[q][0], ow[q][1], ow[q][2], ow[q][3]);
        }
        if (fused) {  // norm of the previous item's x in these columns, before x is overwritten
          float xv[8], gm[8];
          tc_wait_ld_x8(xr);
#pragma unroll
          for (int e = 0; e < 8; ++e) xv[e] = __uint_as_float(xr[e]);
          unpack8(gv, gm);
          uint4 nv;
          nv.x = pack_bf16x2(xv[0] * rprev * gm[0], xv[1] * rprev * gm[1]);
          nv.y = pack_bf16x2(xv[2] * rprev * gm[2], xv[3] * rprev * gm[3]);
          nv.z = pack_bf16x2(xv[4] * rprev * gm[4], xv[5] * rprev * gm[5]);
          nv.w = pack_bf16x2(xv[6] * rprev * gm[6], xv[7] * rprev * gm[7]);
          *reinterpret_cast<uint4*>(ost + kOffNormT + off) = nv;
        }
        tc_st_x8(xaddr + 16 * (sb + c), x);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->out_full[o]);
        if (!MS && i > 0 && c == 0 && warp < 4 && !(ok = read_d(i - 1, nprev))) break;
        if (MS && c > 0 && !(ok = mma_chunk(j - 1, ji - 2))) break;
      }
      if (!ok) break;
      if (KCL == 16 && i > 0 && ni == 0) {  // no columns here (a narrow H): only consume the phases
        if (fused && !(ok = take_rstd(i - 1, prevblk))) break;
        if (!MS && warp < 4 && !(ok = read_d(i - 1, nprev))) break;
      }
      if (MS && ni > 0 && !(ok = mma_chunk(j - 1, ji - 1))) break;
      tc_wait_st();
      // the next item (published an item ahead: usually here already)
      if (!(ok = arrived_warp(i + 1))) break;
      const int nblk = iblock(i + 1);

      // ------------- item finish: hand the partials to the exchange warp --
      const int par = i & 1;
      // the exchange warp has read item i - 2's partials from this slot
      if (i >= 2 && !(ok = wait_warp(X, &tl->red_free[par], ((i >> 1) & 1) ^ 1))) break;
      tl->red[par][warp][lane] = make_float2(sR2.x + sR2.y, sx2.x + sx2.y);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tl->red_full[par]);
        // the item's gate buffer may now be refilled (for item i + 2): no read
        // of it can still be pending, however the gates were kept or re-read
        mbar_arrive(&tl->gates_empty[i & 1]);
      }
      // no MMA follows the last item: its D is read now
      if (!MS && nblk < 0 && warp < 4 && !(ok = read_d(i, ni))) break;
      if (MS) {  // warps w and w + 4 both hold stream w % 4: fold them into dbuf[w % 4]
        const int g = lane >> 2, t4 = lane & 3;
        if (warp >= 4) {
          if (!(ok = wait_warp(X, &tl->dbuf_free, (i & 1) ^ 1))) break;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int n = 0; n < 3; ++n) {
              float* r0 = &tl->dbuf[warp - 4][16 * m + g][8 * n + 2 * t4];
              r0[0] = acc[m][n][0];
              r0[1] = acc[m][n][1];
              r0[8 * kDPad] = acc[m][n][2];
              r0[8 * kDPad + 1] = acc[m][n][3];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&tl->fold_full);
        } else {
          if (!(ok = wait_warp(X, &tl->fold_full, i & 1))) break;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int n = 0; n < 3; ++n) {
              float* r0 = &tl->dbuf[warp][16 * m + g][8 * n + 2 * t4];
              r0[0] += acc[m][n][0];
              r0[1] += acc[m][n][1];
              r0[8 * kDPad] += acc[m][n][2];
              r0[8 * kDPad + 1] += acc[m][n][3];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&tl->dbuf_full);
        }
      }
      if (!full) {
        ++nu;
        sbu += ni;
      }

      // ------------- normalise-only passes: the norm tiles of a group of
      // chunks per output stage (a whole block followed by a unit or by
      // nothing; after the last item, every unit once its block is complete)
      const int qa = full ? -1 : 0, qb = full ? (nblk < 0 || iunit(i + 1) >= 0 ? 0 : -1) : (nblk < 0 ? nu : 0);
      constexpr int NG = G::kNormGroup;
      int sq = 0;  // first tensor-memory slot of the pass's x
      for (int q = qa; q < qb && ok; ++q) {
        const Item u = !SPLIT || q < 0 ? item(i) : const_cast<const Item&>(tl->ulist[q]);
        if (!SPLIT || q < 0) {
          if (!(ok = take_rstd(i, u.block))) break;
        } else {
          const float2 sxo = unit_sx(X, W, u.unit / k_parts, k_parts, kCl, lane);
          if (!(ok = sxo.y != 0.f)) break;
          const int64_t tt = (int64_t)u.block * kBM + lane;
          rprev = tt < T ? 1.0f / sqrtf(sxo.x / (float)H + a.eps) : 0.f;
        }
        const int nq = nchi(u), gq = u.g0;
        for (int c0 = 0; c0 < nq; c0 += NG, ++j) {
          const int o = j % kNO;
          if (!(ok = wait_warp(X, &tl->out_empty[o], ((j / kNO) & 1) ^ 1))) break;
          uint8_t* ost = sm + kOffOut + o * kOutStage;
          const int ng = min(NG, nq - c0);
          for (int g = 0; g < ng; ++g) {
            const int c = c0 + g;
            uint32_t xr[8];
            tc_ld_x8_issue(xaddr + 16 * (sq + c), xr);
            const uint4 gv = gamma8(gq + c);
            tc_wait_ld_x8(xr);
            float xv[8], gm[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = __uint_as_float(xr[e]);
            unpack8(gv, gm);
            uint4 nv;
            nv.x = pack_bf16x2(xv[0] * rprev * gm[0], xv[1] * rprev * gm[1]);
            nv.y = pack_bf16x2(xv[2] * rprev * gm[2], xv[3] * rprev * gm[3]);
            nv.z = pack_bf16x2(xv[4] * rprev * gm[4], xv[5] * rprev * gm[5]);
            nv.w = pack_bf16x2(xv[6] * rprev * gm[6], xv[7] * rprev * gm[7]);
            *reinterpret_cast<uint4*>(ost + g * kRTile + off) = nv;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tl->out_full[o]);
          if (MS) {  // the warp-level projection warps count in the stage's release
            __syncwarp();
            if (lane == 0) mbar_arrive(&tl->out_empty[o]);
          }
        }
        if (q >= 0) sq += nq;
      }
      prevblk = full ? iblock(i) : -1;
      nprev = ni;
      __syncwarp();
      if (lane == 0) {
        release(i);
        if (ok && nblk < 0) release(i + 1);  // the end of the list
      }
    }
    // no tensor-memory load or store of this warp is outstanding at exit
    tc_wait_ld();
    tc_wait_st();
  }

  tc_fence_before();
  __syncwarp();
  // No CTA leaves while a peer may still write into it: every CTA arrives here
  // after its last send, and the cluster barrier's release/acquire orders the
  // peers' stores into this CTA before it goes on.
  cluster_sync_all();
  if (tid == 0 && *X.reported) atomicOr(a.status, 2u);  // a wait of this CTA ran past the limit
  if (*X.aborted) {
    // A CTA that abandoned the call may not have seen every partial a peer
    // sent it arrive on its barriers: before its shared memory is released it
    // also waits a fixed 20 us, far longer than a store into a cluster peer
    // takes to land.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 20000) {
    }
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Kernel pointers of one SCHED setting (form: 0 no_post, 1 post, 2 identity;
// out: 0 bf16, 1 mxfp8, 2 fp8_grid; clusters of 16 run only the tcgen05
// projection).
template <int FORM, bool MS, int KCL, int SCHED>
inline void* stream_kptr_f(int out) {
  return out == 2 ? (void*)stream_seam_kernel<FORM, 2, MS, KCL, SCHED>
         : out == 1 ? (void*)stream_seam_kernel<FORM, 1, MS, KCL, SCHED>
                    : (void*)stream_seam_kernel<FORM, 0, MS, KCL, SCHED>;
}
template <bool MS, int KCL, int SCHED>
inline void* stream_kptr_(int form, int out) {
  return form == 2 ? stream_kptr_f<2, MS, KCL, SCHED>(out)
         : form == 1 ? stream_kptr_f<1, MS, KCL, SCHED>(out) : stream_kptr_f<0, MS, KCL, SCHED>(out);
}
template <int SCHED>
inline void* stream_kernel_ptr_t(int form, int out, bool ms, int kcl) {
  if (kcl == 16) return stream_kptr_<false, 16, SCHED>(form, out);
  return ms ? stream_kptr_<true, 4, SCHED>(form, out) : stream_kptr_<false, 4, SCHED>(form, out);
}

}  // namespace mhc
