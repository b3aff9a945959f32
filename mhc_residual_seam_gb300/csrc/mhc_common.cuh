// Shared device code of the GB300 delayed mHC seam: argument block, bf16 and
// e4m3 helpers, the per-token gate finish and the ue8m0 exponent rule.
//
// The seam ("[FlyDSL] Single-launch Mega-mHC on gfx950", Motivation and
// Kernel Architecture): post-mix -> collapse with the carried pre -> sum of
// squares + 24-logit gate projection -> split-K reduce -> rstd -> sigmoid
// gates and Sinkhorn comb -> layer input RMSNorm -> optional per-32 ue8m0 FP8.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mhc {

constexpr int kStreams = 4;   // n_hc residual streams
constexpr int kLogits = 24;   // 4 pre + 4 post + 16 comb
constexpr int kParts = 26;    // per-token partial sums: 24 logits, sum R'^2, sum x^2
constexpr int kPartStride = 32;

struct SeamArgs {
  const __nv_bfloat16* R;          // [T,4,H]
  const __nv_bfloat16* Y;          // [T,H] or null (no_post)
  const float* post_prev;          // [T,4] or null
  const float* comb_prev;          // [T,4,4]
  const float* pre_prev;           // [T,4]
  const float* fn;                 // [4H,24]
  const __nv_bfloat16* fn_packed;  // [48,4H] hi/lo, or null
  const float* bias;               // [24]
  const float* alpha;              // [3]
  const __nv_bfloat16* gamma;      // [H]
  float eps;
  int64_t T;
  int H;
  __nv_bfloat16* res_out;          // [T,4,H]
  __nv_bfloat16* norm;             // [T,H]
  uint8_t* codes;                  // [T,H]   (mxfp8)
  uint8_t* scales;                 // [T,H/32] (mxfp8)
  __nv_bfloat16* grid;             // [T,H]   (fp8_grid: the quantisation dequantised to bf16)
  float* pre_out;                  // [T,4]
  float* post_out;                 // [T,4]
  float* comb_out;                 // [T,4,4]
  unsigned* status;                // device status word (bit 0: a bounded wait ran out)
  int sinkhorn_iters;
  float amax_floor;
  long long spin_limit;
  int unshifted;                   // 1: the unshifted ordering (x with the fresh pre, no norm; into `norm`)
};

// ------------------------------------------------------------------ bf16 --
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two floats -> packed bf16x2 (round to nearest even); `a` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 bf16pair(uint32_t u) { return make_float2(bf16lo(u), bf16hi(u)); }

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// ------------------------------------------------------------- streaming --
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, const uint4& v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// ----------------------------------------------------------------- ue8m0 --
// Shared exponent of a 32-group: the smallest integer e with
// amax <= 448 * 2^e, from the fp32 bits of max(amax, floor) (exact integer
// logic: 448 = 1.75 * 2^8, so e = E - 135 when the significand is <= 1.75 and
// E - 134 above it), clamped to [-127, 127].
__device__ __forceinline__ int ue8m0_exponent(float amax, float floor_) {
  float a = fmaxf(amax, floor_);
  uint32_t u = __float_as_uint(a);
  int E = (int)((u >> 23) & 0xFF);
  uint32_t f = u & 0x7FFFFFu;
  if (E == 0) {  // fp32 subnormal (only with a tiny floor): renormalise
    int p = 31 - __clz((int)f);
    f = (f << (23 - p)) & 0x7FFFFFu;
    E = p - 22;
  }
  int e = E - 135 + (f > 0x600000u ? 1 : 0);
  return max(-127, min(127, e));
}

// 2^-e as an fp32 (e in [-127, 127] -> normal or the one subnormal 2^-127).
__device__ __forceinline__ float exp2_neg(int e) {
  int b = 127 - e;
  return b > 0 ? __uint_as_float((uint32_t)b << 23) : __uint_as_float(0x00400000u);
}

// Two floats -> two e4m3fn codes, round to nearest even, saturating finite.
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Quantise 32 bf16 norm values (packed 2 per word, 16 words) of one group:
// returns the e8m0 byte, writes 32 codes as 8 words.
__device__ __forceinline__ uint8_t quant_group32(const uint32_t* nb, uint32_t* codes, float floor_) {
  float amax = 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(nb[q])), fabsf(bf16hi(nb[q]))));
  int e = ue8m0_exponent(amax, floor_);
  float s = exp2_neg(e);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint16_t lo = e4m3x2(__fmul_rn(bf16lo(nb[2 * q]), s), __fmul_rn(bf16hi(nb[2 * q]), s));
    uint16_t hi = e4m3x2(__fmul_rn(bf16lo(nb[2 * q + 1]), s), __fmul_rn(bf16hi(nb[2 * q + 1]), s));
    codes[q] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return (uint8_t)(e + 127);
}

// 2^e as an fp32 (e in [-127, 127] -> normal or the one subnormal 2^-127).
__device__ __forceinline__ float exp2_pos(int e) {
  return e > -127 ? __uint_as_float((uint32_t)(127 + e) << 23) : __uint_as_float(0x00400000u);
}

// fp8_grid of one 32-group: the ue8m0 exponent and e4m3 codes as in
// quant_group32, then each code's value times 2^e rounded to bf16 (the e4m3
// value is exact in fp16 and the product by a power of two is exact in fp32
// unless it leaves the range).  Writes 32 bf16 values as 16 words.
__device__ __forceinline__ void grid_group32(const uint32_t* nb, uint32_t* gw, float floor_) {
  float amax = 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(nb[q])), fabsf(bf16hi(nb[q]))));
  const int e = ue8m0_exponent(amax, floor_);
  const float s = exp2_neg(e), up = exp2_pos(e);
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const uint16_t c2 = e4m3x2(__fmul_rn(bf16lo(nb[q]), s), __fmul_rn(bf16hi(nb[q]), s));
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c2, __NV_E4M3);
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    gw[q] = pack_bf16x2(__fmul_rn(v.x, up), __fmul_rn(v.y, up));
  }
}

// ---------------------------------------------------------------- finish --
// Hardware reciprocal (rcp.approx.ftz.f32, within about 1 ulp): the shortest
// dependent step of the Sinkhorn chain.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Gate finish of one token from its reduced partial sums (s_R over 4H, the
// 24 projections d[k]).  Logit order [pre 0..3 | post 4..7 | comb 8..23
// row-major], alpha[0] pre, alpha[1] post, alpha[2] comb.  The Sinkhorn runs
// on exp(l - rowmax): the row scale cancels in the first row normalisation.
// Reciprocals, the exponentials and the reciprocal square root use the fast
// hardware forms (__expf, rsqrtf: a few ulp): the 160 normalisations of the
// Sinkhorn are a serial chain per token on the launch's latency path, the
// accurate forms cost several times the instructions (the finish is inlined
// in every streaming kernel variant), and the gates are checked to 1e-3.
__device__ __forceinline__ void finish_gates(float sR, const float* d, const float* alpha,
                                             const float* bias, int K, float eps, int iters,
                                             float* pre, float* post, float* comb) {
  float rstdR = rsqrtf(sR / (float)K + eps);
  float a0 = alpha[0] * rstdR, a1 = alpha[1] * rstdR, a2 = alpha[2] * rstdR;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    pre[i] = rcp_approx(1.0f + __expf(-(a0 * d[i] + bias[i])));
    post[i] = 2.0f * rcp_approx(1.0f + __expf(-(a1 * d[4 + i] + bias[4 + i])));
  }
  float M[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float l[4], mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      l[j] = a2 * d[8 + 4 * i + j] + bias[8 + 4 * i + j];
      mx = fmaxf(mx, l[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) M[4 * i + j] = __expf(l[j] - mx);
  }
  // (kept rolled: each iteration depends on the last, so unrolling buys no
  // overlap, only instruction footprint)
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float s = rcp_approx((M[4 * i] + M[4 * i + 1]) + (M[4 * i + 2] + M[4 * i + 3]));
#pragma unroll
      for (int j = 0; j < 4; ++j) M[4 * i + j] *= s;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float s = rcp_approx((M[j] + M[4 + j]) + (M[8 + j] + M[12 + j]));
#pragma unroll
      for (int i = 0; i < 4; ++i) M[4 * i + j] *= s;
    }
  }
#pragma unroll
  for (int q = 0; q < 16; ++q) comb[q] = M[q];
}

__device__ __forceinline__ void store_gates(const SeamArgs& a, int64_t t, const float* pre,
                                            const float* post, const float* comb) {
  float4* po = reinterpret_cast<float4*>(a.pre_out + t * 4);
  float4* qo = reinterpret_cast<float4*>(a.post_out + t * 4);
  float4* co = reinterpret_cast<float4*>(a.comb_out + t * 16);
  po[0] = make_float4(pre[0], pre[1], pre[2], pre[3]);
  qo[0] = make_float4(post[0], post[1], post[2], post[3]);
#pragma unroll
  for (int i = 0; i < 4; ++i) co[i] = make_float4(comb[4 * i], comb[4 * i + 1], comb[4 * i + 2], comb[4 * i + 3]);
}

// ------------------------------------------------------- memory ordering --
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

}  // namespace mhc
