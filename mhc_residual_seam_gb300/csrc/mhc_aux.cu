// Auxiliary kernels of libmhcseam: the fn hi/lo pack, the standalone ue8m0
// quantiser, the streaming copy used as the bandwidth ceiling, and the second
// pass of the unshifted ordering.

#include "mhc_common.cuh"

namespace mhc {

// fn [4H, 24] fp32 -> packed [48, 4H] bf16: row k = bf16(fn[:, k]) ("hi"),
// row 24 + k = bf16(fn[:, k] - hi) ("lo").  One thread per row r of fn.
__global__ void pack_fn_kernel(const float* __restrict__ fn, __nv_bfloat16* __restrict__ out, int K) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= K) return;
#pragma unroll
  for (int k = 0; k < kLogits; ++k) {
    float w = fn[(size_t)r * kLogits + k];
    __nv_bfloat16 hi = __float2bfloat16_rn(w);
    __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
    out[(size_t)k * K + r] = hi;
    out[(size_t)(kLogits + k) * K + r] = lo;
  }
}

// Standalone per-32 ue8m0 quantiser: one thread per (row, group).
__global__ void quant_ue8m0_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int H, float floor_,
                                   uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int G = H / 32;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * G) return;
  const int64_t r = idx / G;
  const int g = (int)(idx - r * G);
  const uint4* src = reinterpret_cast<const uint4*>(x + r * H + (int64_t)g * 32);
  uint32_t nb[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 v = __ldcs(src + q);
    nb[4 * q] = v.x; nb[4 * q + 1] = v.y; nb[4 * q + 2] = v.z; nb[4 * q + 3] = v.w;
  }
  uint32_t cw[8];
  uint8_t sb = quant_group32(nb, cw, floor_);
  uint4* dst = reinterpret_cast<uint4*>(codes + r * H + (int64_t)g * 32);
  __stcs(dst, make_uint4(cw[0], cw[1], cw[2], cw[3]));
  __stcs(dst + 1, make_uint4(cw[4], cw[5], cw[6], cw[7]));
  scales[r * G + g] = sb;
}

// Grid-stride 16-byte copy with streaming (evict-first) loads and stores,
// four loads in flight per thread.
__global__ void __launch_bounds__(512) copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
          d = __ldcs(src + i + 3 * stride);
    __stcs(dst + i, a);
    __stcs(dst + i + stride, b);
    __stcs(dst + i + 2 * stride, c);
    __stcs(dst + i + 3 * stride, d);
  }
  for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// The unshifted ordering's second pass on the streaming path: x[t,h] =
// bf16(sum_i pre[t,i] R'[t,i,h]) with the fresh pre the seam kernel just wrote
// (it needs every column's projection, so it follows that kernel on the same
// stream; the recent part of R' is still in L2).  Work item = (token, 8
// columns): four 16-byte R' loads and one 16-byte store, grid-stride.
__global__ void __launch_bounds__(256) unshifted_x_kernel(const __nv_bfloat16* __restrict__ rp,
                                                          const float* __restrict__ pre, int64_t T, int H,
                                                          __nv_bfloat16* __restrict__ x) {
  const int segs = H / 8;
  const int64_t n = T * segs;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t t = i / segs;
    const int h = (int)(i - t * segs) * 8;
    const float4 p = __ldg(reinterpret_cast<const float4*>(pre + t * 4));
    const __nv_bfloat16* r = rp + t * kStreams * H + h;
    float r0[8], r1[8], r2[8], r3[8], xv[8];
    unpack8(__ldcs(reinterpret_cast<const uint4*>(r)), r0);
    unpack8(__ldcs(reinterpret_cast<const uint4*>(r + H)), r1);
    unpack8(__ldcs(reinterpret_cast<const uint4*>(r + 2 * H)), r2);
    unpack8(__ldcs(reinterpret_cast<const uint4*>(r + 3 * H)), r3);
#pragma unroll
    for (int e = 0; e < 8; ++e) xv[e] = fmaf(p.w, r3[e], fmaf(p.z, r2[e], fmaf(p.y, r1[e], p.x * r0[e])));
    uint4 ov;
    ov.x = pack_bf16x2(xv[0], xv[1]); ov.y = pack_bf16x2(xv[2], xv[3]);
    ov.z = pack_bf16x2(xv[4], xv[5]); ov.w = pack_bf16x2(xv[6], xv[7]);
    __stcs(reinterpret_cast<uint4*>(x + t * H + h), ov);
  }
}

cudaError_t unshifted_x_launch(const void* rp, const float* pre, int64_t T, int H, void* x, int num_sms,
                               cudaStream_t s) {
  const int64_t n = T * (H / 8);
  int64_t blocks = (int64_t)num_sms * 8;
  const int64_t need = (n + 255) / 256;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  unshifted_x_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(rp), pre, T, H,
                                                      reinterpret_cast<__nv_bfloat16*>(x));
  return cudaGetLastError();
}

cudaError_t pack_fn_launch(const float* fn, void* out, int H, cudaStream_t s) {
  const int K = kStreams * H;
  pack_fn_kernel<<<(K + 255) / 256, 256, 0, s>>>(fn, reinterpret_cast<__nv_bfloat16*>(out), K);
  return cudaGetLastError();
}

cudaError_t quant_launch(const void* x, int64_t rows, int H, float floor_, uint8_t* codes, uint8_t* scales,
                         cudaStream_t s) {
  const int64_t n = rows * (H / 32);
  const int64_t blocks = (n + 255) / 256;
  quant_ue8m0_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x), rows, H, floor_,
                                                      codes, scales);
  return cudaGetLastError();
}

cudaError_t copy_launch(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  size_t blocks = (size_t)num_sms * 4;
  const size_t need = (n16 + 511) / 512;
  if (blocks > need) blocks = need;
  if (blocks == 0) blocks = 1;
  copy_kernel<<<(unsigned)blocks, 512, 0, s>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

}  // namespace mhc
