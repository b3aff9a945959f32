// C ABI of libmhcseam: argument checks, launch policy, per-device set-up and
// dispatch to the seam kernels.  See include/mhc_seam.h for the contract.

#include <mutex>
#include <string>

#include "mhc_common.cuh"
#include "../../include/mhc_seam.h"

namespace mhc {
// mhc_split.cu
using SplitKernel = void (*)(SeamArgs, int, int, int64_t, char*, size_t);
size_t split_slot_bytes(int Gh, int BT);
size_t split_smem_bytes(int BT, int Wd, bool unshifted);
cudaError_t split_init(size_t max_smem);
cudaError_t split_capacity(bool post, int mode, int BT, int Wd, int num_sms, int* ctas);
cudaError_t split_launch(const SeamArgs& a, int BT, int Wd, int64_t groups_per_launch, char* slots,
                         cudaStream_t stream, int* launches);
// mhc_stream.cu
cudaError_t stream_init();
int stream_cols(int H);
bool stream_tc_fits(int H);
cudaError_t stream_launch(const SeamArgs& a, bool tcgen05_proj, int kcl, cudaStream_t stream,
                          unsigned long long report_ns, int* launches, void* wsx, int wave_split);
size_t stream_split_bytes();
int stream_last_parts();
// mhc_aux.cu
cudaError_t pack_fn_launch(const float* fn, void* out, int H, cudaStream_t s);
cudaError_t quant_launch(const void* x, int64_t rows, int H, float floor_, uint8_t* codes, uint8_t* scales,
                         cudaStream_t s);
cudaError_t copy_launch(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t s);
cudaError_t unshifted_x_launch(const void* rp, const float* pre, int64_t T, int H, void* x, int num_sms,
                               cudaStream_t s);
}  // namespace mhc

namespace {

constexpr size_t kHeaderBytes = 256;  // status word + padding, at the start of every workspace
constexpr long long kDefaultSpin = 10000000LL;
constexpr int kMaxDevices = 64;
constexpr size_t kSplitMaxSmem = 160 * 1024;
constexpr int64_t kStreamMinT = 1024;  // auto policy: clusters of 4 from this many tokens, of 16 below

thread_local std::string g_err;
thread_local int g_launches = 0;
thread_local int g_last_parts_api = 1;

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorString(e);
  return MHC_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device one-time set-up (kernel attributes, SM count).  Refused while the
// stream is capturing, because the attribute calls are not stream work.
int ensure_device(cudaStream_t stream, DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MHC_ERR_CUDA, "device index out of range");
  DeviceState& st = g_dev[dev];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!st.ready) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
      return fail(MHC_ERR_CAPTURE, "the first call on a device must not be made during stream capture");
    e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = mhc::split_init(kSplitMaxSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute (split path)");
    e = mhc::stream_init();
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute (streaming path)");
    st.ready = true;
  }
  *out = &st;
  return MHC_OK;
}

struct Plan {
  int path = 1;          // 1 split, 2 streaming (clusters of 4), 3 streaming (clusters of 16)
  bool tc_proj = false;  // streaming path: tcgen05 projection instead of warp-level MMA
  int BT = 8;   // tokens per CTA (split path)
  int Wd = 64;  // columns per CTA (split path)
};

int next_pow2(int64_t v) {
  int p = 1;
  while (p < v && p < 32) p <<= 1;
  return p;
}

// Launch policy: a pure function of (T, H, cfg, whether fn_packed is given,
// the ordering).  Workspace sizing asks with and without fn_packed and takes
// the larger, so a workspace sized for the automatic policy fits whichever
// path the call takes.  The unshifted ordering takes the same paths (on
// the streaming path as two launches) but needs twice the split path's shared
// memory per CTA.
int make_plan(int64_t T, int H, const mhc_config* cfg, bool have_packed, Plan* p, bool unshifted = false) {
  mhc_config c = {};
  if (cfg) c = *cfg;
  if (c.path < 0 || c.path > 3) return fail(MHC_ERR_CONFIG, "cfg.path must be 0, 1, 2 or 3");
  if (c.block_m != 0 && (c.block_m < 0 || c.block_m > 32 || (c.block_m & (c.block_m - 1)) != 0))
    return fail(MHC_ERR_CONFIG, "cfg.block_m must be 0 or a power of two <= 32");
  if (c.cols_per_cta != 0 && (c.cols_per_cta < 32 || c.cols_per_cta % 32 != 0 || c.cols_per_cta > 16384))
    return fail(MHC_ERR_CONFIG, "cfg.cols_per_cta must be 0 or a multiple of 32 in [32, 16384]");
  if (c.sinkhorn_iters < 0 || c.sinkhorn_iters > 10000) return fail(MHC_ERR_CONFIG, "cfg.sinkhorn_iters out of range");
  if (!(c.amax_floor >= 0.f) || c.amax_floor > 1e30f) return fail(MHC_ERR_CONFIG, "cfg.amax_floor out of range");
  if (c.spin_limit < 0) return fail(MHC_ERR_CONFIG, "cfg.spin_limit must be >= 0");
  if (c.projection < 0 || c.projection > 2) return fail(MHC_ERR_CONFIG, "cfg.projection must be 0, 1 or 2");
  if (c.wave_split < 0 || c.wave_split > 64) return fail(MHC_ERR_CONFIG, "cfg.wave_split must be in [0, 64]");
  const bool stream_ok = mhc::stream_cols(H) > 0;
  p->path = c.path;
  if (p->path == 0) {  // a split-path knob (block_m, cols_per_cta) picks the split path
    if (!stream_ok || c.block_m || c.cols_per_cta) p->path = 1;
    else if (T >= kStreamMinT) p->path = 2;
    else p->path = (H >= 1024 && have_packed) ? 3 : 1;
  }
  if (p->path == 2 || p->path == 3) {
    if (!stream_ok) return fail(MHC_ERR_SHAPE, "the streaming path needs H a multiple of 64 with 512 <= H <= 8192");
    if (p->path == 3) {  // at most 8 chunks per CTA: the tcgen05 projection always fits
      if (c.projection == 1)
        return fail(MHC_ERR_CONFIG, "the streaming path with clusters of 16 runs the tcgen05 projection only");
      p->tc_proj = true;
      return MHC_OK;
    }
    p->tc_proj = c.projection == 2 || (c.projection == 0 && mhc::stream_tc_fits(H));
    if (c.projection == 2 && !mhc::stream_tc_fits(H))
      return fail(MHC_ERR_CONFIG, "the tcgen05 projection needs H <= 5120 (tensor memory holds x and the accumulator)");
    return MHC_OK;
  }
  if (T <= 8) {
    p->BT = next_pow2(T < 1 ? 1 : T);
    p->Wd = 64;
  } else if (T <= 32) {
    p->BT = 8;
    p->Wd = 128;
  } else if (T <= 128) {
    p->BT = 16;
    p->Wd = 256;
  } else {
    p->BT = 32;
    p->Wd = 320;
  }
  if (c.block_m) p->BT = c.block_m;
  if (c.cols_per_cta) p->Wd = c.cols_per_cta;
  const int Hr = (H + 31) / 32 * 32;
  if (p->Wd > Hr) p->Wd = Hr;
  if (mhc::split_smem_bytes(p->BT, p->Wd, unshifted) > kSplitMaxSmem)
    return fail(MHC_ERR_CONFIG, "block_m * cols_per_cta too large: x of one CTA does not fit in shared memory");
  return MHC_OK;
}

size_t plan_workspace(int64_t T, int H, const Plan& p) {
  if (p.path != 1) return kHeaderBytes + mhc::stream_split_bytes();  // status word + the split partial round
  const int Gh = (H + p.Wd - 1) / p.Wd;
  const int64_t groups = (T + p.BT - 1) / p.BT;
  return kHeaderBytes + mhc::split_slot_bytes(Gh, p.BT) * (size_t)(groups > 0 ? groups : 1);
}

struct Range {
  uintptr_t lo, hi;
};
Range rng(const void* p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

}  // namespace

extern "C" {

// The policy may pick another path when fn_packed is given: size for both.
static size_t workspace_for(int64_t T, int H, const mhc_config* cfg, bool unshifted) {
  Plan p, q;
  if (T < 0 || H <= 0 || make_plan(T, H, cfg, false, &p, unshifted) != MHC_OK) return kHeaderBytes;
  size_t n = plan_workspace(T, H, p);
  if (make_plan(T, H, cfg, true, &q, unshifted) == MHC_OK) {
    const size_t m = plan_workspace(T, H, q);
    if (m > n) n = m;
  }
  return n;
}

size_t mhc_workspace_bytes(int64_t T, int H, const mhc_config* cfg) { return workspace_for(T, H, cfg, false); }

size_t mhc_workspace_bytes_unshifted(int64_t T, int H, const mhc_config* cfg) {
  return workspace_for(T, H, cfg, true);
}

int mhc_workspace_init(void* ws, size_t bytes, void* stream) {
  if (!ws || bytes < kHeaderBytes) return fail(MHC_ERR_WORKSPACE, "workspace NULL or too small");
  cudaError_t e = cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MHC_OK : cuda_fail(e, "cudaMemsetAsync");
}

int mhc_check_status(void* ws, void* stream) {
  if (!ws) return fail(MHC_ERR_WORKSPACE, "workspace NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (v == 0) return MHC_OK;
  e = cudaMemsetAsync(ws, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  return fail(MHC_ERR_TIMEOUT, "a bounded device wait ran out in an earlier call on this workspace");
}

size_t mhc_packed_fn_bytes(int H) { return H > 0 ? (size_t)2 * mhc::kLogits * mhc::kStreams * (size_t)H * 2 : 0; }

int mhc_pack_fn(const float* fn, void* fn_packed, int H, void* stream) {
  if (!fn || !fn_packed) return fail(MHC_ERR_NULL, "fn and fn_packed are required");
  if (H <= 0 || H % 8 != 0) return fail(MHC_ERR_SHAPE, "H must be a positive multiple of 8");
  if (!aligned16(fn) || !aligned16(fn_packed)) return fail(MHC_ERR_ALIGN, "fn and fn_packed must be 16-byte aligned");
  cudaError_t e = mhc::pack_fn_launch(fn, fn_packed, H, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MHC_OK : cuda_fail(e, "pack_fn launch");
}

// Both orderings: `unsh` selects the unshifted one (then pre_prev and gamma
// are NULL, out_mode is bf16, and `norm` receives x).
static int seam_impl(bool unsh, const void* R, const void* Y, const float* post_prev, const float* comb_prev,
                     const float* pre_prev, const float* fn, const void* fn_packed, const float* bias,
                     const float* alpha, const void* gamma, float eps, int64_t T, int H, mhc_out_mode out_mode,
                     void* residual_out, void* norm, uint8_t* fp8_codes, uint8_t* e8m0_scales, float* pre_out,
                     float* post_out, float* comb_out, void* workspace, size_t ws_bytes, const mhc_config* cfg,
                     void* stream) {
  g_launches = 0;
  g_last_parts_api = 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (out_mode != MHC_OUT_BF16 && out_mode != MHC_OUT_MXFP8 && out_mode != MHC_OUT_FP8_GRID)
    return fail(MHC_ERR_CONFIG, "unknown out_mode");
  const bool mx = out_mode == MHC_OUT_MXFP8, gridm = out_mode == MHC_OUT_FP8_GRID;
  if (T < 0 || H <= 0 || H % 8 != 0) return fail(MHC_ERR_SHAPE, "need T >= 0 and H a positive multiple of 8");
  if ((mx || gridm) && H % 32 != 0) return fail(MHC_ERR_SHAPE, "mxfp8 and fp8_grid outputs need H % 32 == 0");
  if (!(eps >= 0.f) || eps > 1e30f) return fail(MHC_ERR_CONFIG, "eps must be finite and >= 0");
  Plan plan;
  int rc = make_plan(T, H, cfg, fn_packed != nullptr, &plan, unsh);
  if (rc != MHC_OK) return rc;
  if (T == 0) return MHC_OK;
  if ((Y == nullptr) != (post_prev == nullptr))
    return fail(MHC_ERR_INCOMPLETE_POST, "Y and post_prev must both be given (post form) or both be NULL (no_post)");
  // comb_prev NULL: the identity (first-block) form, R' = R; residual_out is
  // not written (and may be NULL)
  const bool ident = comb_prev == nullptr;
  if (ident && Y) return fail(MHC_ERR_INCOMPLETE_POST, "the identity form (comb_prev NULL) takes no Y and no post_prev");
  if (ident) residual_out = nullptr;
  if (!R || (!unsh && (!pre_prev || !gamma)) || !fn || !bias || !alpha || (!ident && !residual_out) || !norm ||
      !pre_out || !post_out || !comb_out)
    return fail(MHC_ERR_NULL, "a required pointer is NULL");
  if (mx && (!fp8_codes || !e8m0_scales)) return fail(MHC_ERR_NULL, "mxfp8 output needs fp8_codes and e8m0_scales");
  if (gridm && !fp8_codes) return fail(MHC_ERR_NULL, "fp8_grid output needs fp8_codes (the bf16 grid)");
  if (gridm && plan.path == 1)
    return fail(MHC_ERR_CONFIG, "fp8_grid runs on the streaming path (cfg.path 2 or 3, fn_packed, 512 <= H <= 8192)");
  if (!workspace) return fail(MHC_ERR_WORKSPACE, "workspace is NULL");
  const void* a16[] = {R, Y, post_prev, comb_prev, pre_prev, fn, fn_packed, gamma, residual_out, norm,
                       (mx || gridm) ? fp8_codes : nullptr, pre_out, post_out, comb_out, workspace};
  for (const void* p : a16)
    if (p && !aligned16(p)) return fail(MHC_ERR_ALIGN, "a pointer that must be 16-byte aligned is not");
  if (reinterpret_cast<uintptr_t>(bias) % 4 || reinterpret_cast<uintptr_t>(alpha) % 4)
    return fail(MHC_ERR_ALIGN, "bias and alpha must be 4-byte aligned");
  const size_t need = plan_workspace(T, H, plan);
  if (ws_bytes < need) return fail(MHC_ERR_WORKSPACE, "workspace smaller than mhc_workspace_bytes(T, H, cfg)");

  // Overlap checks: outputs against inputs (R' may be R exactly) and each other.
  const size_t TH = (size_t)T * H;
  Range in[] = {rng(R, TH * 8), rng(Y, Y ? TH * 2 : 0), rng(post_prev, post_prev ? (size_t)T * 16 : 0),
                rng(comb_prev, comb_prev ? (size_t)T * 64 : 0), rng(pre_prev, pre_prev ? (size_t)T * 16 : 0), rng(fn, (size_t)H * 4 * 24 * 4),
                rng(fn_packed, fn_packed ? mhc_packed_fn_bytes(H) : 0), rng(bias, 96), rng(alpha, 12),
                rng(gamma, gamma ? (size_t)H * 2 : 0)};
  Range out[] = {rng(residual_out, residual_out ? TH * 8 : 0), rng(norm, TH * 2), rng(fp8_codes, mx ? TH : (gridm ? TH * 2 : 0)),
                 rng(e8m0_scales, mx ? TH / 32 : 0), rng(pre_out, (size_t)T * 16), rng(post_out, (size_t)T * 16),
                 rng(comb_out, (size_t)T * 64), rng(workspace, need)};
  const int n_in = sizeof in / sizeof in[0], n_out = sizeof out / sizeof out[0];
  for (int o = 0; o < n_out; ++o) {
    for (int i = 0; i < n_in; ++i) {
      if (o == 0 && i == 0 && residual_out == R) continue;  // in-place post-mix
      if (overlap(out[o], in[i])) return fail(MHC_ERR_ALIAS, "an output overlaps an input");
    }
    for (int q = o + 1; q < n_out; ++q)
      if (overlap(out[o], out[q])) return fail(MHC_ERR_ALIAS, "two outputs overlap");
  }

  DeviceState* dev = nullptr;
  rc = ensure_device(s, &dev);
  if (rc != MHC_OK) return rc;

  mhc::SeamArgs a;
  a.R = static_cast<const __nv_bfloat16*>(R);
  a.Y = static_cast<const __nv_bfloat16*>(Y);
  a.post_prev = post_prev;
  a.comb_prev = comb_prev;
  a.pre_prev = pre_prev;
  a.fn = fn;
  a.fn_packed = static_cast<const __nv_bfloat16*>(fn_packed);
  a.bias = bias;
  a.alpha = alpha;
  a.gamma = static_cast<const __nv_bfloat16*>(gamma);
  a.eps = eps;
  a.T = T;
  a.H = H;
  a.res_out = static_cast<__nv_bfloat16*>(residual_out);
  a.norm = static_cast<__nv_bfloat16*>(norm);
  a.codes = mx ? fp8_codes : nullptr;
  a.scales = mx ? e8m0_scales : nullptr;
  a.grid = gridm ? reinterpret_cast<__nv_bfloat16*>(fp8_codes) : nullptr;
  a.pre_out = pre_out;
  a.post_out = post_out;
  a.comb_out = comb_out;
  a.status = static_cast<unsigned*>(workspace);
  a.sinkhorn_iters = (cfg && cfg->sinkhorn_iters) ? cfg->sinkhorn_iters : 20;
  a.amax_floor = (cfg && cfg->amax_floor > 0.f) ? cfg->amax_floor : 1e-10f;
  a.spin_limit = (cfg && cfg->spin_limit) ? cfg->spin_limit : kDefaultSpin;
  a.unshifted = unsh ? 1 : 0;

  int launches = 0;
  if (plan.path == 2 || plan.path == 3) {
    if (!fn_packed) return fail(MHC_ERR_NULL, "the streaming path needs fn_packed (mhc_pack_fn) or cfg.path = 1");
    if (T >= ((int64_t)1 << 31)) return fail(MHC_ERR_SHAPE, "the streaming path takes T < 2^31");
    mhc::SeamArgs a1 = a;
    if (unsh) {
      // First pass of the unshifted ordering: R', the gates and the fresh pre.
      // Its x and norm are not stored (norm NULL); the carried pre and gamma
      // that feed them are pointed at R, which is valid memory of at least
      // T * 16 and H * 2 bytes, so the discarded arithmetic reads no stray
      // address.
      a1.norm = nullptr;
      a1.gamma = a.R;
      a1.pre_prev = reinterpret_cast<const float*>(a.R);
      a1.unshifted = 0;
    }
    cudaError_t e = mhc::stream_launch(a1, plan.tc_proj, plan.path == 3 ? 16 : 4, s,
                                       (unsigned long long)a.spin_limit * 100ull, &launches,
                                       static_cast<char*>(workspace) + kHeaderBytes, cfg ? cfg->wave_split : 0);
    if (e == cudaErrorInvalidValue) return fail(MHC_ERR_CUDA, "tensor map encoding failed (streaming path)");
    if (e != cudaSuccess) return cuda_fail(e, "seam launch (streaming path)");
    g_last_parts_api = mhc::stream_last_parts();
    if (unsh) {  // second pass: x = sum_i pre[i] R'[i] with the fresh pre
      e = mhc::unshifted_x_launch(ident ? R : residual_out, pre_out, T, H, norm, dev->num_sms, s);
      if (e != cudaSuccess) return cuda_fail(e, "x launch (unshifted ordering)");
      ++launches;
    }
    g_launches = launches;
    return MHC_OK;
  }
  int cap = 0;
  cudaError_t e = mhc::split_capacity(Y != nullptr, unsh ? 2 : (mx ? 1 : 0), plan.BT, plan.Wd, dev->num_sms, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query (split path)");
  const int Gh = (H + plan.Wd - 1) / plan.Wd;
  int64_t per_launch = cap / Gh;
  if (per_launch < 1) return fail(MHC_ERR_CONFIG, "cols_per_cta too small: one token group does not fit on the GPU");
  e = mhc::split_launch(a, plan.BT, plan.Wd, per_launch, static_cast<char*>(workspace) + kHeaderBytes, s, &launches);
  if (e != cudaSuccess) return cuda_fail(e, "seam launch (split path)");
  g_launches = launches;
  return MHC_OK;
}

int mhc_seam(const void* R, const void* Y, const float* post_prev, const float* comb_prev, const float* pre_prev,
             const float* fn, const void* fn_packed, const float* bias, const float* alpha, const void* gamma,
             float eps, int64_t T, int H, mhc_out_mode out_mode, void* residual_out, void* norm, uint8_t* fp8_codes,
             uint8_t* e8m0_scales, float* pre_out, float* post_out, float* comb_out, void* workspace,
             size_t ws_bytes, const mhc_config* cfg, void* stream) {
  return seam_impl(false, R, Y, post_prev, comb_prev, pre_prev, fn, fn_packed, bias, alpha, gamma, eps, T, H,
                   out_mode, residual_out, norm, fp8_codes, e8m0_scales, pre_out, post_out, comb_out, workspace,
                   ws_bytes, cfg, stream);
}

int mhc_seam_unshifted(const void* R, const void* Y, const float* post_prev, const float* comb_prev,
                       const float* fn, const void* fn_packed, const float* bias, const float* alpha, float eps,
                       int64_t T, int H, void* residual_out, void* x_out, float* pre_out, float* post_out,
                       float* comb_out, void* workspace, size_t ws_bytes, const mhc_config* cfg, void* stream) {
  return seam_impl(true, R, Y, post_prev, comb_prev, nullptr, fn, fn_packed, bias, alpha, nullptr, eps, T, H,
                   MHC_OUT_BF16, residual_out, x_out, nullptr, nullptr, pre_out, post_out, comb_out, workspace,
                   ws_bytes, cfg, stream);
}

int mhc_quant_ue8m0(const void* x, int64_t rows, int H, float amax_floor, uint8_t* codes, uint8_t* scales,
                    void* stream) {
  if (rows < 0 || H <= 0 || H % 32 != 0) return fail(MHC_ERR_SHAPE, "need rows >= 0 and H a positive multiple of 32");
  if (rows == 0) return MHC_OK;
  if (!x || !codes || !scales) return fail(MHC_ERR_NULL, "x, codes and scales are required");
  if (!aligned16(x) || !aligned16(codes)) return fail(MHC_ERR_ALIGN, "x and codes must be 16-byte aligned");
  const size_t n = (size_t)rows * H;
  if (overlap(rng(x, n * 2), rng(codes, n)) || overlap(rng(x, n * 2), rng(scales, n / 32)) ||
      overlap(rng(codes, n), rng(scales, n / 32)))
    return fail(MHC_ERR_ALIAS, "buffers overlap");
  cudaError_t e = mhc::quant_launch(x, rows, H, amax_floor > 0.f ? amax_floor : 1e-10f, codes, scales,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MHC_OK : cuda_fail(e, "quant launch");
}

int mhc_copy(const void* src, void* dst, size_t bytes, void* stream) {
  if (bytes == 0) return MHC_OK;
  if (!src || !dst) return fail(MHC_ERR_NULL, "src and dst are required");
  if (!aligned16(src) || !aligned16(dst) || bytes % 16) return fail(MHC_ERR_ALIGN, "16-byte aligned pointers and sizes");
  if (overlap(rng(src, bytes), rng(dst, bytes))) return fail(MHC_ERR_ALIAS, "src and dst overlap");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  e = mhc::copy_launch(src, dst, bytes, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MHC_OK : cuda_fail(e, "copy launch");
}

int mhc_last_launch_count(void) { return g_launches; }

int mhc_last_wave_parts(void) { return g_last_parts_api; }

const char* mhc_last_error_string(void) { return g_err.c_str(); }

}  // extern "C"

namespace mhc {
void set_last_error(const std::string& msg) { g_err = msg; }
}  // namespace mhc
