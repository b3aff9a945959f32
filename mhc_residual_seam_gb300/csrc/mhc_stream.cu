// Streaming path of the delayed mHC seam: bandwidth-tuned for large T.
//
// One cluster of 8 CTAs per block of 32 tokens; CTA r of the cluster owns
// columns [r W, (r+1) W) of H for all four streams (W = H / 8).  Per 64-column
// chunk, TMA brings the four R tiles, the Y tile and the four hi/lo-packed fn
// tiles into shared memory (128-byte swizzle); eight compute warps (thread =
// token, warp = 8-column slice) post-mix in fp32, round R' to bf16 in place,
// accumulate the sums of squares, and store the collapsed x in tensor memory;
// one thread issues the gate projection on the tensor cores (tcgen05,
// D[64 x 32] += fn^T[64 x 64] . R'^T[64 x 32] per stream and 16-wide k step,
// rows 0..23 hi, 24..47 lo, fp32 accumulation in TMEM) and stores R' with TMA.
// The split over the 8 CTAs is reduced through distributed shared memory:
// each CTA sends its per-token partials to the token's owner CTA, the owner
// finishes the gates and sends rstd_x back, and every CTA normalises its own
// x from tensor memory ("[FlyDSL] Single-launch Mega-mHC on gfx950", Kernel
// Architecture: split-K, DIST_FINISH -- here co-residency is guaranteed by
// the cluster launch, so no wait can depend on an unscheduled CTA).
//
// Roles: warps 0-7 compute, warp 8 TMA producer, warp 9 MMA issuer, R' store
// and tensor-memory owner.  Two pipeline stages; two CTAs per SM.

#include <cooperative_groups.h>

#include "mhc_common.cuh"
#include "mhc_sm100.cuh"

namespace cg = cooperative_groups;

namespace mhc {

// Gate finish of one token on its owner CTA, kept out of line so its arrays
// do not raise the register pressure of the streaming loop.
__device__ __noinline__ void finish_owner(const SeamArgs& a, int64_t t, const float* p, int H, float* r) {
  float pre[4], post[4], cb[16];
  finish_gates(p[24], p, a.alpha, a.bias, kStreams * H, a.eps, a.sinkhorn_iters, pre, post, cb);
  store_gates(a, t, pre, post, cb);
  *r = 1.0f / sqrtf(p[25] / (float)H + a.eps);
}
constexpr int kClusterCtas = 8;
constexpr int kBM = 32;                 // tokens per cluster
constexpr int kChunk = 64;              // columns per pipeline stage
constexpr int kStreamThreads = 320;     // 8 compute warps + producer + MMA
constexpr int kFnRows = 48;             // 24 hi + 24 lo
constexpr uint32_t kFnTile = kFnRows * 128;    // 6 KB
constexpr uint32_t kRTile = kBM * 128;         // 4 KB
constexpr uint32_t kOffFn = 0;
constexpr uint32_t kOffR = 4 * kFnTile;        // 24 KB
constexpr uint32_t kOffY = kOffR + 4 * kRTile; // 40 KB
constexpr uint32_t kStageBytes = kOffY + kRTile;  // 44 KB
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColD = 0;           // D: 32 columns (tokens)
constexpr uint32_t kColX = 32;          // x: 16 columns per chunk
constexpr int kMaxChunks = (int)((kTmemCols - kColX) / 16);  // 14
constexpr uint32_t kIdesc = idesc_bf16_f32(64, kBM);

struct StreamTail {
  uint64_t full[2], rdy[2], empty[2], dfull, drained;
  uint32_t tmem_base;
  int err;
  float red[8][kBM][2];       // per compute warp: sum R'^2, sum x^2 of each token
  float dmat[kFnRows][kBM];   // D rows (hi 0..23, lo 24..47) x tokens
  float recv[kClusterCtas][kBM / kClusterCtas][kParts];  // partials sent to this owner CTA
  float rstd[kBM];            // rstd_x of the block's tokens
};

size_t stream_smem_bytes() { return 2 * kStageBytes + sizeof(StreamTail) + 1024; }

__device__ __forceinline__ void note_timeout(const SeamArgs& a, StreamTail* tl) {
  tl->err = 1;
  atomicOr(a.status, 2u);
}

template <bool POST, bool MXFP8>
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kStreamThreads, 2)
    stream_seam_kernel(const SeamArgs a, const __grid_constant__ CUtensorMap tmR,
                       const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmRo,
                       const __grid_constant__ CUtensorMap tmFn, const __grid_constant__ CUtensorMap tmN,
                       const __grid_constant__ CUtensorMap tmC, int W, unsigned long long limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage0 = sm;
  StreamTail* tl = reinterpret_cast<StreamTail*>(sm + 2 * kStageBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int H = a.H;
  const int64_t T = a.T;
  const int64_t t0 = (int64_t)(blockIdx.x / kClusterCtas) * kBM;
  const int hbase = rank * W;
  const int wcols = max(0, min(W, H - hbase));
  const int nch = (wcols + kChunk - 1) / kChunk;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tl->full[s], 1);
      mbar_init(&tl->rdy[s], 8);
      mbar_init(&tl->empty[s], 2);
    }
    mbar_init(&tl->dfull, 1);
    mbar_init(&tl->drained, 1);
    tl->err = 0;
    mbar_fence_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tmR);
    prefetch_tmap(&tmFn);
    if (POST) prefetch_tmap(&tmY);
    prefetch_tmap(&tmRo);
  }
  if (warp == 9) {
    tmem_alloc(&tl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster.sync();  // barriers initialised; every CTA of the cluster is running
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      const uint64_t pol_stream = l2_evict_first(), pol_w = l2_evict_last();
      const uint32_t bytes = 4 * kFnTile + 4 * kRTile + (POST ? kRTile : 0);
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        const uint32_t ph = (c >> 1) & 1;
        if (!mbar_wait(&tl->empty[s], ph ^ 1, limit_ns)) {
          note_timeout(a, tl);
          break;
        }
        uint8_t* st = stage0 + s * kStageBytes;
        const int h = hbase + c * kChunk;
        mbar_arrive_expect_tx(&tl->full[s], bytes);
#pragma unroll
        for (int i = 0; i < 4; ++i) tma_load_3d(st + kOffFn + i * kFnTile, &tmFn, &tl->full[s], h, i, 0, pol_w);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          tma_load_3d(st + kOffR + i * kRTile, &tmR, &tl->full[s], h, i, (int)t0, pol_stream);
        if (POST) tma_load_2d(st + kOffY, &tmY, &tl->full[s], h, (int)t0, pol_stream);
        issued = c + 1;
      }
      // Every load this CTA issued has landed before it can exit (bounded;
      // immediate unless a consumer gave up waiting).
      for (int c = (issued > 2 ? issued - 2 : 0); c < issued; ++c)
        if (!mbar_wait(&tl->full[c & 1], (c >> 1) & 1, limit_ns)) note_timeout(a, tl);
    }
  } else if (warp == 9) {
    // -------------------------------------- MMA issuer and R' tile store --
    if (lane == 0) {
      for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        const uint32_t ph = (c >> 1) & 1;
        if (!mbar_wait(&tl->rdy[s], ph, limit_ns)) {
          note_timeout(a, tl);
          break;
        }
        tc_fence_after();
        uint8_t* st = stage0 + s * kStageBytes;
        const uint32_t fa = smem_u32(st + kOffFn), rb = smem_u32(st + kOffR);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc_mma_bf16(tmem + kColD, sdesc_k_sw128(fa + i * kFnTile + kk * 32), sdesc_k_sw128(rb + i * kRTile + kk * 32),
                        kIdesc, (c | i | kk) != 0);
          }
        }
        tc_commit(&tl->empty[s]);
        const int h = hbase + c * kChunk;
#pragma unroll
        for (int i = 0; i < 4; ++i) tma_store_3d(&tmRo, st + kOffR + i * kRTile, h, i, (int)t0);
        tma_store_commit();
        tma_store_wait_read_all();
        mbar_arrive(&tl->empty[s]);
      }
      tc_commit(&tl->dfull);
      mbar_arrive(&tl->drained);
      tma_store_wait_all();
    }
  } else {
    // ------------------------------------------------------- compute warps --
    const int q = warp & 3, wq = warp >> 2;
    const int64_t t = t0 + lane;
    const bool tv = t < T;
    float comb[16], postg[4], preg[4];
#pragma unroll
    for (int k = 0; k < 16; ++k) comb[k] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) postg[k] = preg[k] = 0.f;
    if (tv) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float4 v = __ldg(reinterpret_cast<const float4*>(a.comb_prev + t * 16) + k);
        comb[4 * k] = v.x; comb[4 * k + 1] = v.y; comb[4 * k + 2] = v.z; comb[4 * k + 3] = v.w;
      }
      float4 p = __ldg(reinterpret_cast<const float4*>(a.pre_prev + t * 4));
      preg[0] = p.x; preg[1] = p.y; preg[2] = p.z; preg[3] = p.w;
      if (POST) {
        float4 v = __ldg(reinterpret_cast<const float4*>(a.post_prev + t * 4));
        postg[0] = v.x; postg[1] = v.y; postg[2] = v.z; postg[3] = v.w;
      }
    }
    const uint32_t xaddr = tmem + ((uint32_t)(32 * q) << 16) + kColX + 8 * wq;
    const uint32_t off = lane * 128 + ((warp ^ (lane & 7)) << 4);  // row = token, 16-byte chunk = warp
    float sR = 0.f, sx = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int s = c & 1;
      const uint32_t ph = (c >> 1) & 1;
      if (!mbar_wait(&tl->full[s], ph, limit_ns)) {
        note_timeout(a, tl);
        break;
      }
      uint8_t* st = stage0 + s * kStageBytes;
      // inputs stay packed (bf16x2 words); one word = two columns at a time
      uint4 rin[4], yin = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < 4; ++j) rin[j] = *reinterpret_cast<const uint4*>(st + kOffR + j * kRTile + off);
      if (POST) yin = *reinterpret_cast<const uint4*>(st + kOffY + off);
      uint32_t ow[4][4];
      float x[8];
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        const uint32_t w0 = (&rin[0].x)[wd], w1 = (&rin[1].x)[wd], w2 = (&rin[2].x)[wd], w3 = (&rin[3].x)[wd];
        const uint32_t wy = (&yin.x)[wd];
        const float a0 = bf16lo(w0), a1 = bf16lo(w1), a2 = bf16lo(w2), a3 = bf16lo(w3), ya = bf16lo(wy);
        const float b0 = bf16hi(w0), b1 = bf16hi(w1), b2 = bf16hi(w2), b3 = bf16hi(w3), yb = bf16hi(wy);
        float xa = 0.f, xb = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float va = comb[4 * i] * a0, vb = comb[4 * i] * b0;
          va = fmaf(comb[4 * i + 1], a1, va); vb = fmaf(comb[4 * i + 1], b1, vb);
          va = fmaf(comb[4 * i + 2], a2, va); vb = fmaf(comb[4 * i + 2], b2, vb);
          va = fmaf(comb[4 * i + 3], a3, va); vb = fmaf(comb[4 * i + 3], b3, vb);
          if (POST) { va = fmaf(postg[i], ya, va); vb = fmaf(postg[i], yb, vb); }
          const uint32_t o = pack_bf16x2(va, vb);
          ow[i][wd] = o;
          const float ra = bf16lo(o), rb = bf16hi(o);
          sR = fmaf(ra, ra, sR);
          sR = fmaf(rb, rb, sR);
          xa = fmaf(preg[i], ra, xa);
          xb = fmaf(preg[i], rb, xb);
        }
        x[2 * wd] = xa;
        x[2 * wd + 1] = xb;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(st + kOffR + i * kRTile + off) = make_uint4(ow[i][0], ow[i][1], ow[i][2], ow[i][3]);
#pragma unroll
      for (int e = 0; e < 8; ++e) sx = fmaf(x[e], x[e], sx);
      tc_st_x8(xaddr + 16 * c, x);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->rdy[s]);
    }
    tc_wait_st();
    tl->red[warp][lane][0] = sR;
    tl->red[warp][lane][1] = sx;
  }

  // ---------------------------------------------------- partial sums out --
  __syncthreads();
  if (warp < 4) {
    float dv[32];
    bool ok = nch > 0 && mbar_wait(&tl->dfull, 0, limit_ns);
    if (nch > 0 && !ok) note_timeout(a, tl);
    tc_fence_after();
    if (ok) {
      // M = 64 accumulator: row m sits in lane 32 (m / 16) + m % 16
      const uint32_t daddr = tmem + ((uint32_t)(32 * warp) << 16) + kColD;
#pragma unroll
      for (int k = 0; k < 4; ++k) tc_ld_x8(daddr + 8 * k, dv + 8 * k);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) dv[k] = 0.f;
    }
    const int m = 16 * warp + lane;
    if (lane < 16 && m < kFnRows) {
#pragma unroll
      for (int n = 0; n < kBM; ++n) tl->dmat[m][n] = dv[n];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < kBM * kParts; idx += kStreamThreads) {
    const int tok = idx / kParts, k = idx - tok * kParts;
    float v;
    if (k < 24) {
      v = tl->dmat[k][tok] + tl->dmat[24 + k][tok];
    } else {
      v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += tl->red[w][tok][k - 24];
    }
    float* dst = cluster.map_shared_rank(&tl->recv[rank][tok / kClusterCtas][k], tok % kClusterCtas);
    *dst = v;
  }
  cluster.sync();

  // ---------------------------------------- owner: gates and rstd_x -----
  if (tid < kBM / kClusterCtas) {
    const int tok = rank + kClusterCtas * tid;
    const int64_t t = t0 + tok;
    float p[kParts];
#pragma unroll
    for (int k = 0; k < kParts; ++k) {
      float s = 0.f;
#pragma unroll
      for (int src = 0; src < kClusterCtas; ++src) s += tl->recv[src][tid][k];
      p[k] = s;
    }
    float r = 0.f;
    if (t < T) {
      finish_owner(a, t, p, H, &r);
    }
    for (int dst = 0; dst < kClusterCtas; ++dst) *cluster.map_shared_rank(&tl->rstd[tok], dst) = r;
  }
  cluster.sync();

  // --------------------------------------------------------------- norm --
  uint8_t* nbuf = stage0;                       // nch x [32 x 64] bf16, 128-byte swizzle
  uint8_t* cbuf = stage0 + kMaxChunks * kRTile; // nch x [32 x 64] u8, row-major
  if (warp < 8) {
    if (!mbar_wait(&tl->drained, 0, limit_ns)) note_timeout(a, tl);
    const int q = warp & 3, wq = warp >> 2;
    const uint32_t xaddr = tmem + ((uint32_t)(32 * q) << 16) + kColX + 8 * wq;
    const uint32_t off = lane * 128 + ((warp ^ (lane & 7)) << 4);
    const float r = tl->rstd[lane];
    for (int c = 0; c < nch; ++c) {
      float x[8], gm[8];
      tc_ld_x8(xaddr + 16 * c, x);
      const int h = hbase + c * kChunk + 8 * warp;
      if (h < H) {
        unpack8(__ldg(reinterpret_cast<const uint4*>(a.gamma + h)), gm);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) gm[e] = 0.f;
      }
      uint4 ov;
      ov.x = pack_bf16x2(x[0] * r * gm[0], x[1] * r * gm[1]);
      ov.y = pack_bf16x2(x[2] * r * gm[2], x[3] * r * gm[3]);
      ov.z = pack_bf16x2(x[4] * r * gm[4], x[5] * r * gm[5]);
      ov.w = pack_bf16x2(x[6] * r * gm[6], x[7] * r * gm[7]);
      *reinterpret_cast<uint4*>(nbuf + c * kRTile + off) = ov;
    }
  }
  __syncthreads();
  if (MXFP8) {
    // one thread per (token, 32-column group): the group's amax and codes
    for (int idx = tid; idx < kBM * nch * 2; idx += kStreamThreads) {
      const int tok = idx % kBM, grp = idx / kBM;
      const int c = grp >> 1, half = grp & 1;
      const int h = hbase + c * kChunk + 32 * half;
      uint32_t nb[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ch = 4 * half + j;
        uint4 v = *reinterpret_cast<const uint4*>(nbuf + c * kRTile + tok * 128 + ((ch ^ (tok & 7)) << 4));
        nb[4 * j] = v.x; nb[4 * j + 1] = v.y; nb[4 * j + 2] = v.z; nb[4 * j + 3] = v.w;
      }
      uint32_t cw[8];
      const uint8_t sb = quant_group32(nb, cw, a.amax_floor);
      uint4* cd = reinterpret_cast<uint4*>(cbuf + c * (kBM * 64) + tok * 64 + 32 * half);
      cd[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      cd[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
      const int64_t t = t0 + tok;
      if (t < T && h < H) a.scales[t * (H / 32) + h / 32] = sb;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    for (int c = 0; c < nch; ++c) {
      tma_store_2d(&tmN, nbuf + c * kRTile, hbase + c * kChunk, (int)t0);
      if (MXFP8) tma_store_2d(&tmC, cbuf + c * (kBM * 64), hbase + c * kChunk, (int)t0);
    }
    tma_store_commit();
    tma_store_wait_all();
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- host side --
using StreamKernel = void (*)(SeamArgs, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                              CUtensorMap, int, unsigned long long);

static void* stream_kernel_ptr(bool post, bool mxfp8) {
  if (post) return mxfp8 ? (void*)stream_seam_kernel<true, true> : (void*)stream_seam_kernel<true, false>;
  return mxfp8 ? (void*)stream_seam_kernel<false, true> : (void*)stream_seam_kernel<false, false>;
}

cudaError_t stream_init() {
  for (int p = 0; p < 2; ++p)
    for (int m = 0; m < 2; ++m) {
      cudaError_t e = cudaFuncSetAttribute(stream_kernel_ptr(p, m), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)stream_smem_bytes());
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

// Columns per CTA for width H, or 0 when the streaming path cannot take H.
int stream_cols(int H) {
  if (H % kChunk != 0 || H < kChunk * kClusterCtas) return 0;
  const int chunks = (H / kChunk + kClusterCtas - 1) / kClusterCtas;
  if (chunks > kMaxChunks) return 0;
  return chunks * kChunk;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled get_encode() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  }
  return fn;
}

static bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiled enc = get_encode();
  if (!enc) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Returns cudaSuccess, or cudaErrorInvalidValue when a tensor map cannot be
// encoded (the caller reports it).
cudaError_t stream_launch(const SeamArgs& a, cudaStream_t stream, unsigned long long limit_ns, int* launches) {
  const int H = a.H;
  const int W = stream_cols(H);
  if (W == 0) return cudaErrorInvalidValue;
  const cuuint64_t T = (cuuint64_t)a.T;
  CUtensorMap mR, mY, mRo, mFn, mN, mC;
  const cuuint64_t d3[3] = {(cuuint64_t)H, 4, T};
  const cuuint64_t s3[2] = {(cuuint64_t)H * 2, (cuuint64_t)H * 8};
  const cuuint32_t b3[3] = {kChunk, 1, kBM};
  const cuuint64_t d2[2] = {(cuuint64_t)H, T};
  const cuuint64_t s2[1] = {(cuuint64_t)H * 2};
  const cuuint32_t b2[2] = {kChunk, kBM};
  const cuuint64_t dF[3] = {(cuuint64_t)H, 4, kFnRows};
  const cuuint32_t bF[3] = {kChunk, 1, kFnRows};
  const cuuint64_t sC[1] = {(cuuint64_t)H};
  bool ok = encode(&mR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.R, d3, s3, b3, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode(&mRo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.res_out, d3, s3, b3, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode(&mFn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.fn_packed, dF, s3, bF, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode(&mN, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.norm, d2, s2, b2, CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok) ok = encode(&mY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.Y ? (const void*)a.Y : (const void*)a.R, d2, s2, b2,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok) ok = encode(&mC, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.codes ? (const void*)a.codes : (const void*)a.norm, d2,
                      sC, b2, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  const int64_t blocks = (a.T + kBM - 1) / kBM;
  void* k = stream_kernel_ptr(a.Y != nullptr, a.codes != nullptr);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks * kClusterCtas), 1, 1);
  cfg.blockDim = dim3(kStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = stream_smem_bytes();
  cfg.stream = stream;
  int Wi = W;
  void* args[] = {const_cast<SeamArgs*>(&a), &mR, &mY, &mRo, &mFn, &mN, &mC, &Wi, &limit_ns};
  cudaError_t e = cudaLaunchKernelExC(&cfg, k, args);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace mhc
