// Split path of the delayed mHC seam: latency-tuned for small T.
//
// Why this shape: at decode sizes the 4H x 24 fp32 gate weight (1.97 MB at
// H = 5120) is most of what a CTA must read, so H is spread over many small
// CTAs (a few dozen columns each) and every CTA covers all tokens of its
// token group.  The projection runs on the CUDA cores (FFMA); the partial
// sums are reduced across the CTAs of a token group through a global
// workspace, and the last-arriving CTA finishes the gates ("[FlyDSL]
// Single-launch Mega-mHC on gfx950", Kernel Architecture: split-K with a
// last-arriving-workgroup finish; DIST_FINISH: the last arrival publishes rstd
// and every split rescales its own x).  The launch is cooperative, so every
// CTA of the grid is resident and the wait for rstd always ends; the wait is
// also bounded, and a wait that runs out sets bit 0 of the status word.
//
// Grid: (Gh column slices, Gt token groups of BT tokens); 256 threads.
// Work item = (token, 8 consecutive columns): four 16-byte R loads and one Y
// load, the 4x4 post-mix in fp32, one bf16 rounding, and the rounded R' feeds
// the sums, the projection and x (x stays in shared memory until rstd_x).
//
// The unshifted ordering (MODE 2) keeps the CTA's R' in shared memory instead
// of x: the finishing CTA publishes the fresh pre of each token (in place of
// rstd_x), and every CTA then forms its columns of x = sum_i pre[i] R'[i],
// stored as bf16 with no norm.

#include <string>

#include "mhc_common.cuh"

namespace mhc {

constexpr int kSplitThreads = 256;
constexpr int kSplitWarps = kSplitThreads / 32;

// Workspace of one token group (one slot per gridDim.y): arrival counter and
// generation word, rstd_x of the group's tokens, and the per-CTA partials
// [Gh][BT][32] (26 used; in the unshifted ordering words 26-29 of CTA 0's rows
// carry the fresh pre from the finishing CTA to the others).
constexpr size_t kSlotCtrl = 64;
constexpr size_t kSlotRstd = 128;  // 32 floats

size_t split_slot_bytes(int Gh, int BT) {
  size_t b = kSlotCtrl + kSlotRstd + (size_t)Gh * BT * kPartStride * sizeof(float);
  return (b + 255) & ~(size_t)255;
}

constexpr int kPartPre = 26;  // unshifted: the fresh pre in words 26-29 of CTA 0's partial rows

// Dynamic shared memory: x [BT][Wd] fp32 (unshifted: R' [BT][Wd/8][4] of
// 16-byte bf16 runs, twice the bytes), per-warp partials, the finisher's sums.
size_t split_smem_bytes(int BT, int Wd, bool unshifted) {
  return sizeof(float) * ((size_t)BT * Wd * (unshifted ? 2 : 1) + (size_t)kSplitWarps * BT * kParts +
                          (size_t)BT * kParts);
}

// MODE: 0 bf16 norm, 1 bf16 norm + mxfp8, 2 the unshifted ordering
template <bool POST, int MODE, int BT>
__global__ void __launch_bounds__(kSplitThreads) split_seam_kernel(SeamArgs a, int Wd, int Gh,
                                                                   int64_t tok_base, char* slots,
                                                                   size_t slot_bytes) {
  constexpr bool MXFP8 = MODE == 1, UNSH = MODE == 2;
  extern __shared__ float smem[];
  float* xs = smem;                               // [BT][Wd] (unshifted: R' of the four streams)
  float* wp = xs + (size_t)BT * Wd * (UNSH ? 2 : 1);    // [warps][BT][kParts]
  float* tot = wp + (size_t)kSplitWarps * BT * kParts;  // [BT][kParts]
  __shared__ float s_rstd[BT];
  __shared__ float4 s_pre[UNSH ? BT : 1];
  __shared__ int s_last;
  __shared__ unsigned s_gen;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = a.H;
  const int64_t T = a.T;
  const int g = blockIdx.x;
  const int64_t t0 = tok_base + (int64_t)blockIdx.y * BT;
  const int h0 = g * Wd;
  const int wcols = max(0, min(Wd, H - h0));
  const int nseg = wcols >> 3;
  char* slot = slots + (size_t)blockIdx.y * slot_bytes;
  unsigned* ctrl = reinterpret_cast<unsigned*>(slot);
  float* rstd_ws = reinterpret_cast<float*>(slot + kSlotCtrl);
  float* part = reinterpret_cast<float*>(slot + kSlotCtrl + kSlotRstd);

  const int tl = tid % BT;  // every item of this thread belongs to token tl
  const int64_t t = t0 + tl;
  const bool tvalid = t < T;

  // no comb: the identity (first-block) form, R' = R and no residual write
  const bool ident = a.comb_prev == nullptr;
  float comb[16], postg[4], preg[4];
  if (tvalid) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 c = ident ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldg(reinterpret_cast<const float4*>(a.comb_prev + t * 16) + q);
      comb[4 * q] = c.x; comb[4 * q + 1] = c.y; comb[4 * q + 2] = c.z; comb[4 * q + 3] = c.w;
    }
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!UNSH) p = __ldg(reinterpret_cast<const float4*>(a.pre_prev + t * 4));
    preg[0] = p.x; preg[1] = p.y; preg[2] = p.z; preg[3] = p.w;
    if (POST) {
      float4 q = __ldg(reinterpret_cast<const float4*>(a.post_prev + t * 4));
      postg[0] = q.x; postg[1] = q.y; postg[2] = q.z; postg[3] = q.w;
    }
  }

  float acc[kParts];
#pragma unroll
  for (int k = 0; k < kParts; ++k) acc[k] = 0.f;

  if (tvalid) {
    for (int item = tid; item < BT * nseg; item += kSplitThreads) {
      const int seg = item / BT;
      const int h = h0 + seg * 8;
      const __nv_bfloat16* Rt = a.R + (t * kStreams) * H + h;
      float rin[4][8], y[8], x[8];
      uint4 rv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) rv[j] = ld_stream(Rt + (size_t)j * H);
      if (POST) unpack8(ld_stream(a.Y + t * H + h), y);
#pragma unroll
      for (int j = 0; j < 4; ++j) unpack8(rv[j], rin[j]);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float s = comb[4 * i] * rin[0][e];
          s = fmaf(comb[4 * i + 1], rin[1][e], s);
          s = fmaf(comb[4 * i + 2], rin[2][e], s);
          s = fmaf(comb[4 * i + 3], rin[3][e], s);
          if (POST) s = fmaf(postg[i], y[e], s);
          v[e] = s;
        }
        uint4 ov = rv[i];
        if (!ident) {
          ov.x = pack_bf16x2(v[0], v[1]); ov.y = pack_bf16x2(v[2], v[3]);
          ov.z = pack_bf16x2(v[4], v[5]); ov.w = pack_bf16x2(v[6], v[7]);
          st_stream(a.res_out + (t * kStreams + i) * H + h, ov);
        }
        if (UNSH) reinterpret_cast<uint4*>(xs)[((size_t)tl * (Wd >> 3) + seg) * kStreams + i] = ov;
        float rp[8];
        unpack8(ov, rp);
        const float4* f = reinterpret_cast<const float4*>(a.fn + ((size_t)i * H + h) * kLogits);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[24] = fmaf(rp[e], rp[e], acc[24]);
          x[e] = fmaf(preg[i], rp[e], x[e]);
#pragma unroll
          for (int q = 0; q < 6; ++q) {
            float4 w = __ldg(f + e * 6 + q);
            acc[4 * q + 0] = fmaf(rp[e], w.x, acc[4 * q + 0]);
            acc[4 * q + 1] = fmaf(rp[e], w.y, acc[4 * q + 1]);
            acc[4 * q + 2] = fmaf(rp[e], w.z, acc[4 * q + 2]);
            acc[4 * q + 3] = fmaf(rp[e], w.w, acc[4 * q + 3]);
          }
        }
      }
      if (!UNSH) {
        float* xrow = xs + (size_t)tl * Wd + seg * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          xrow[e] = x[e];
          acc[25] = fmaf(x[e], x[e], acc[25]);
        }
      }
    }
  }

  // ---- reduce the partials of this CTA: lanes of one token, then warps ----
#pragma unroll
  for (int k = 0; k < kParts; ++k) {
#pragma unroll
    for (int m = 16; m >= BT; m >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], m);
  }
  if (lane < BT) {
#pragma unroll
    for (int k = 0; k < kParts; ++k) wp[((size_t)warp * BT + lane) * kParts + k] = acc[k];
  }
  __syncthreads();
  for (int idx = tid; idx < BT * kParts; idx += kSplitThreads) {
    const int tt = idx / kParts, k = idx - tt * kParts;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kSplitWarps; ++w) s += wp[((size_t)w * BT + tt) * kParts + k];
    __stcg(part + ((size_t)g * BT + tt) * kPartStride + k, s);
  }
  __threadfence();
  __syncthreads();

  // ---- arrive; the last CTA of the token group finishes ----
  if (tid == 0) {
    unsigned gen0 = ld_acquire_gpu(ctrl + 1);
    unsigned old = atom_add_acq_rel_gpu(ctrl + 0, 1u);
    s_last = (old == (unsigned)(Gh - 1));
    s_gen = gen0;
  }
  __syncthreads();

  if (s_last) {
    if (tid == 0) ctrl[0] = 0u;  // self-reset for the next call on this workspace
    for (int tt = warp; tt < BT; tt += kSplitWarps) {
      if (lane < kParts) {
        float s = 0.f;
        for (int gg = 0; gg < Gh; ++gg) s += __ldcg(part + ((size_t)gg * BT + tt) * kPartStride + lane);
        tot[tt * kParts + lane] = s;
      }
    }
    __syncthreads();
    if (tid < BT) {
      const int64_t tt = t0 + tid;
      float r = 0.f;
      if (tt < T) {
        const float* p = tot + tid * kParts;
        float pre[4], post[4], cb[16];
        finish_gates(p[24], p, a.alpha, a.bias, kStreams * H, a.eps, a.sinkhorn_iters, pre, post, cb);
        store_gates(a, tt, pre, post, cb);
        r = 1.0f / sqrtf(p[25] / (float)H + a.eps);
        if (UNSH) {
          const float4 pv = make_float4(pre[0], pre[1], pre[2], pre[3]);
#pragma unroll
          for (int q = 0; q < 4; ++q) __stcg(part + (size_t)tid * kPartStride + kPartPre + q, (&pv.x)[q]);
          s_pre[tid] = pv;
        }
      } else if (UNSH) {
        s_pre[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __stcg(rstd_ws + tid, r);
      s_rstd[tid] = r;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release_gpu(ctrl + 1, s_gen + 1u);
  } else {
    if (tid == 0) {
      long long n = 0;
      while (ld_acquire_gpu(ctrl + 1) == s_gen) {
        if (++n > a.spin_limit) {
          atomicOr(a.status, 1u);
          break;
        }
        __nanosleep(32);
      }
    }
    __syncthreads();
    if (tid < BT) {
      s_rstd[tid] = __ldcg(rstd_ws + tid);
      if (UNSH) {
        float4 pv;
#pragma unroll
        for (int q = 0; q < 4; ++q) (&pv.x)[q] = __ldcg(part + (size_t)tid * kPartStride + kPartPre + q);
        s_pre[tid] = pv;
      }
    }
  }
  __syncthreads();

  // ---- unshifted: x = sum_i pre[i] R'[i] with the fresh pre, bf16, no norm ----
  if (UNSH) {
    if (tvalid) {
      const float4 pv = s_pre[tl];
      for (int item = tid; item < BT * nseg; item += kSplitThreads) {
        const int seg = item / BT;
        const int h = h0 + seg * 8;
        const uint4* rr = reinterpret_cast<const uint4*>(xs) + ((size_t)tl * (Wd >> 3) + seg) * kStreams;
        float r0[8], r1[8], r2[8], r3[8], xv[8];
        unpack8(rr[0], r0);
        unpack8(rr[1], r1);
        unpack8(rr[2], r2);
        unpack8(rr[3], r3);
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] = fmaf(pv.w, r3[e], fmaf(pv.z, r2[e], fmaf(pv.y, r1[e], pv.x * r0[e])));
        uint4 ov;
        ov.x = pack_bf16x2(xv[0], xv[1]); ov.y = pack_bf16x2(xv[2], xv[3]);
        ov.z = pack_bf16x2(xv[4], xv[5]); ov.w = pack_bf16x2(xv[6], xv[7]);
        st_stream(a.norm + t * H + h, ov);
      }
    }
    return;
  }

  // ---- norm (and the ue8m0 quantiser) of this CTA's columns ----
  if (!MXFP8) {
    if (tvalid) {
      const float r = s_rstd[tl];
      for (int item = tid; item < BT * nseg; item += kSplitThreads) {
        const int seg = item / BT;
        const int h = h0 + seg * 8;
        const float* xrow = xs + (size_t)tl * Wd + seg * 8;
        float gm[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(a.gamma + h)), gm);
        uint4 ov;
        ov.x = pack_bf16x2(xrow[0] * r * gm[0], xrow[1] * r * gm[1]);
        ov.y = pack_bf16x2(xrow[2] * r * gm[2], xrow[3] * r * gm[3]);
        ov.z = pack_bf16x2(xrow[4] * r * gm[4], xrow[5] * r * gm[5]);
        ov.w = pack_bf16x2(xrow[6] * r * gm[6], xrow[7] * r * gm[7]);
        st_stream(a.norm + t * H + h, ov);
      }
    }
  } else {
    const int ngrp = wcols >> 5;
    for (int idx = tid; idx < BT * ngrp; idx += kSplitThreads) {
      const int tl2 = idx % BT, grp = idx / BT;
      const int64_t t2 = t0 + tl2;
      if (t2 >= T) continue;
      const int h = h0 + grp * 32;
      const float r = s_rstd[tl2];
      const float* xrow = xs + (size_t)tl2 * Wd + grp * 32;
      uint32_t nb[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float gm[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(a.gamma + h) + q), gm);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          nb[4 * q + e] = pack_bf16x2(xrow[8 * q + 2 * e] * r * gm[2 * e], xrow[8 * q + 2 * e + 1] * r * gm[2 * e + 1]);
      }
      uint4* nd = reinterpret_cast<uint4*>(a.norm + t2 * H + h);
#pragma unroll
      for (int q = 0; q < 4; ++q) st_stream(nd + q, make_uint4(nb[4 * q], nb[4 * q + 1], nb[4 * q + 2], nb[4 * q + 3]));
      uint32_t cw[8];
      uint8_t sb = quant_group32(nb, cw, a.amax_floor);
      uint4* cd = reinterpret_cast<uint4*>(a.codes + t2 * H + h);
      st_stream(cd, make_uint4(cw[0], cw[1], cw[2], cw[3]));
      st_stream(cd + 1, make_uint4(cw[4], cw[5], cw[6], cw[7]));
      a.scales[t2 * (H / 32) + h / 32] = sb;
    }
  }
}

// ------------------------------------------------------------- launcher --
using SplitKernel = void (*)(SeamArgs, int, int, int64_t, char*, size_t);

template <bool POST, int MODE>
static SplitKernel pick_bt(int BT) {
  switch (BT) {
    case 1: return split_seam_kernel<POST, MODE, 1>;
    case 2: return split_seam_kernel<POST, MODE, 2>;
    case 4: return split_seam_kernel<POST, MODE, 4>;
    case 8: return split_seam_kernel<POST, MODE, 8>;
    case 16: return split_seam_kernel<POST, MODE, 16>;
    case 32: return split_seam_kernel<POST, MODE, 32>;
    default: return nullptr;
  }
}

// mode: 0 bf16 norm, 1 + mxfp8, 2 the unshifted ordering
SplitKernel split_kernel(bool post, int mode, int BT) {
  if (post) return mode == 2 ? pick_bt<true, 2>(BT) : mode == 1 ? pick_bt<true, 1>(BT) : pick_bt<true, 0>(BT);
  return mode == 2 ? pick_bt<false, 2>(BT) : mode == 1 ? pick_bt<false, 1>(BT) : pick_bt<false, 0>(BT);
}

size_t split_workspace_bytes(int Gh, int BT, int64_t groups_per_launch) {
  return split_slot_bytes(Gh, BT) * (size_t)groups_per_launch;
}

// Configure every instantiation once per device (dynamic shared memory cap).
cudaError_t split_init(size_t max_smem) {
  const int bts[] = {1, 2, 4, 8, 16, 32};
  for (int p = 0; p < 2; ++p)
    for (int m = 0; m < 3; ++m)
      for (int b : bts) {
        cudaError_t e = cudaFuncSetAttribute(split_kernel(p, m, b), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)max_smem);
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

// Largest number of CTAs of this instantiation that can be resident at once.
cudaError_t split_capacity(bool post, int mode, int BT, int Wd, int num_sms, int* ctas) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, split_kernel(post, mode, BT), kSplitThreads,
                                                                split_smem_bytes(BT, Wd, mode == 2));
  *ctas = per_sm * num_sms;
  return e;
}

// Launch the split path over tokens [0, T) in waves of at most
// `groups_per_launch` token groups (each wave a cooperative launch).
cudaError_t split_launch(const SeamArgs& a, int BT, int Wd, int64_t groups_per_launch, char* slots,
                         cudaStream_t stream, int* launches) {
  const int Gh = (a.H + Wd - 1) / Wd;
  const size_t slot_bytes = split_slot_bytes(Gh, BT);
  const int64_t groups = (a.T + BT - 1) / BT;
  const int mode = a.unshifted ? 2 : (a.codes != nullptr ? 1 : 0);
  SplitKernel k = split_kernel(a.Y != nullptr, mode, BT);
  for (int64_t g0 = 0; g0 < groups; g0 += groups_per_launch) {
    const int64_t n = groups - g0 < groups_per_launch ? groups - g0 : groups_per_launch;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)Gh, (unsigned)n, 1);
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
    cfg.dynamicSmemBytes = split_smem_bytes(BT, Wd, mode == 2);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, a, Wd, Gh, g0 * BT, slots, slot_bytes);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  return cudaSuccess;
}

}  // namespace mhc
