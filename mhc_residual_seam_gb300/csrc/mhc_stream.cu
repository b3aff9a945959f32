// Streaming path of the delayed mHC seam, host side: kernel variants, tensor
// maps, the wave-edge split policy and the launch.  The kernel itself (and
// its design notes) is in mhc_stream_kernel.cuh; the variants that split the
// partial last round are instantiated in mhc_stream_split.cu.

#include "mhc_stream_kernel.cuh"

namespace mhc {

// The variants with the wave-edge split (mhc_stream_split.cu).
void* stream_kernel_ptr_split(int form, int out, bool ms, int kcl);

// ------------------------------------------------------------- host side --
// form: 0 no_post, 1 post, 2 identity.  Clusters of 16 run only the tcgen05
// projection (at most 8 chunks per CTA).  sched: 0 static, 1 tickets (only
// the bf16 post and no_post forms on clusters of 4 with the tcgen05
// projection: there a cluster's drift costs more than the larger code;
// nullptr elsewhere), 2 tickets and the split.
static void* stream_kernel_ptr(int form, int out, bool ms, int kcl, int sched) {
  if (sched == 2) return stream_kernel_ptr_split(form, out, ms, kcl);
  if (sched == 1) {
    if (out != 0 || ms || kcl != 4 || form == 2) return nullptr;
    return form == 1 ? (void*)stream_seam_kernel<1, 0, false, 4, 1> : (void*)stream_seam_kernel<0, 0, false, 4, 1>;
  }
  return stream_kernel_ptr_t<0>(form, out, ms, kcl);
}
// lean: the identity form with the tcgen05 projection (its own layout)
template <bool L>
static size_t smem_bytes_t(int kcl, int out) {
  if (kcl == 16)
    return out == 2 ? Geo<16, 2, L>::kSmemBytes : out == 1 ? Geo<16, 1, L>::kSmemBytes : Geo<16, 0, L>::kSmemBytes;
  return out == 2 ? Geo<4, 2, L>::kSmemBytes : out == 1 ? Geo<4, 1, L>::kSmemBytes : Geo<4, 0, L>::kSmemBytes;
}
static size_t smem_bytes(int kcl, int out, int form, bool ms) {
  return form == 2 && !ms ? smem_bytes_t<true>(kcl, out) : smem_bytes_t<false>(kcl, out);
}

cudaError_t stream_init() {
  for (int p = 0; p < 3; ++p)          // form
    for (int m = 0; m < 3; ++m)        // out mode
      for (int v = 0; v < 9; ++v) {    // v % 3: 0 tcgen05 / 4, 1 warp MMA / 4, 2 tcgen05 / 16; v / 3: sched
        const int kcl = v % 3 == 2 ? 16 : 4;
        void* k = stream_kernel_ptr(p, m, v % 3 == 1, kcl, v / 3);
        if (k == nullptr) continue;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_bytes(kcl, m, p, v % 3 == 1));
        if (e == cudaSuccess && kcl == 16) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

// Most columns one CTA handles at width H (its chunk count times 64), or 0
// when the streaming path cannot take H.
int stream_cols(int H) {
  if (H % kChunk != 0 || H < 512) return 0;
  const int chunks = (H / kChunk + 3) / 4;
  if (chunks > kMaxChunks) return 0;
  return chunks * kChunk;
}

// Whether the tcgen05 projection fits: its accumulator and x share the 512
// tensor-memory columns.
bool stream_tc_fits(int H) {
  const int W = stream_cols(H);
  return W > 0 && W / kChunk <= kMaxChunksTC;
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

// Clusters that fit at once, per device and kernel variant (queried once).
static int max_clusters(int form, int out, bool ms, int kcl, int sched) {
  static int cache[81][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int v = form + 3 * out + 9 * (kcl == 16 ? 2 : (ms ? 1 : 0)) + 27 * sched;
  if (cache[v][dev] > 0) return cache[v][dev];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)kcl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)kcl, 1, 1);
  cfg.blockDim = dim3(out == 2 ? threads_of<2>() : threads_of<0>(), 1, 1);
  cfg.dynamicSmemBytes = smem_bytes(kcl, out, form, ms);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  void* kp = stream_kernel_ptr(form, out, ms, kcl, sched);
  if (kp == nullptr || cudaOccupancyMaxActiveClusters(&n, kp, &cfg) != cudaSuccess) return 0;
  cache[v][dev] = n;
  return n;
}

// Column parts per block of the last streaming launch's partial round on this
// host thread (1: no split).
thread_local int g_last_parts = 1;
int stream_last_parts() { return g_last_parts; }

// Bytes of the global workspace the split partial round uses (after the
// status header of the caller's workspace).
size_t stream_split_bytes() { return kSplitCntBytes + (kSplitSxFloats + kSplitPpFloats) * sizeof(float); }

// Column parts per block of the last R = n_blocks mod ncl blocks (1: no
// split).  Cut into k parts, those blocks take about ceil(k R / ncl) units of
// ceil(G / k) chunk steps on the busiest cluster (G column groups per CTA)
// instead of G, but each part carries a fixed cost: the normalise-only pass of
// the cluster's last whole block, the global exchange of s_x and of the
// projections, the wait for the other parts and the owner's gate finish.
// Measured on GB300 at H = 5120 that cost is about 24 chunk steps, more than a
// whole block's 20, so the policy (`force` 0) does not split; k >= 2 asks for
// at most k parts where they fit, 1 never splits.  The clusters together must
// hold every unit: each holds at most kMaxUnitsCl of them and at most cap
// tensor-memory chunks of them (their x stays there until the cluster's last
// item); whole column groups only.
static int wave_parts(int n_blocks, int ncl, int n64, int kcl, bool tc_proj, int force) {
  if (force <= 1 || n64 % kcl != 0 || ncl <= 0) return 1;
  const int G = n64 / kcl, R = n_blocks % ncl;
  if (R == 0 || G < 2 || R > kMaxSplitBlocks) return 1;
  const int cap = tc_proj ? kMaxChunksTC : kMaxChunks;
  auto fits = [&](int k) {
    const int maxng = (G + k - 1) / k;
    const int per_cl = cap / maxng < kMaxUnitsCl ? cap / maxng : kMaxUnitsCl;
    return k * R <= kMaxUnits && (long long)per_cl * ncl >= (long long)k * R;
  };
  for (int k = force < G ? force : G; k >= 2; --k)
    if (fits(k)) return k;
  return 1;
}

static cudaError_t launch_with_maps(const SeamArgs& a, const CUtensorMap* m, bool tcgen05_proj, int kcl,
                                    cudaStream_t stream, unsigned long long report_ns, int* launches, void* wsx,
                                    int wave_split);
static cudaError_t launch_range(const SeamArgs& a, const CUtensorMap* m, bool tcgen05_proj, int kcl, int block0,
                                int n_blocks, cudaStream_t stream, unsigned long long report_ns, int* launches,
                                void* wsx, int wave_split);

// Returns cudaSuccess, or cudaErrorInvalidValue when a tensor map cannot be
// encoded or no cluster fits (the caller reports it).  kcl: CTAs per cluster
// (4, or 16 with the tcgen05 projection).
// report_ns: a device wait longer than this sets status bit 1 and goes on; a
// wait one second longer than that abandons the call (the kernel stops issuing
// work, drains what is in flight and returns).  wsx: stream_split_bytes() of
// zeroed device memory (counters reset themselves after each call).
// wave_split: parts per block of the partial last round (0 policy, 1 none).
cudaError_t stream_launch(const SeamArgs& a, bool tcgen05_proj, int kcl, cudaStream_t stream,
                          unsigned long long report_ns, int* launches, void* wsx, int wave_split) {
  const int H = a.H;
  if (stream_cols(H) == 0 || (kcl != 4 && kcl != 16) || (kcl == 16 && !tcgen05_proj)) return cudaErrorInvalidValue;
  const cuuint64_t T = (cuuint64_t)a.T;
  // The nine tensor maps depend only on the buffers, (T, H) and the output
  // mode (the quantised-output map is bf16 with 2H-byte rows for the fp8_grid
  // and u8 with H-byte rows for mxfp8, on possibly the same buffer): a caller
  // that repeats a call with the same buffers and mode (a decode loop) reuses
  // them instead of encoding them again on the host.
  struct MapSet {
    const void* key[9];
    int64_t T;
    int H;
    int out;
    CUtensorMap m[9];
  };
  thread_local MapSet cache[4];
  thread_local int cache_next = 0;
  const int out_mode = a.grid ? 2 : a.codes ? 1 : 0;
  const void* key[9] = {a.R, a.Y, a.res_out, a.fn_packed, a.norm, a.grid ? (const void*)a.grid : (const void*)a.codes,
                        a.comb_prev, a.pre_prev, a.post_prev};
  for (const MapSet& c : cache) {
    bool hit = c.T == a.T && c.H == H && c.out == out_mode;
    for (int i = 0; hit && i < 9; ++i) hit = c.key[i] == key[i];
    if (hit) return launch_with_maps(a, c.m, tcgen05_proj, kcl, stream, report_ns, launches, wsx, wave_split);
  }
  CUtensorMap mR, mY, mRo, mFn, mN, mC;
  // R and R' [T, 4, H] as (column, token, stream) and the packed fn
  // [48, 4H] as (column, row, stream): one box carries the four streams'
  // tiles of a chunk, laid out in shared memory stream by stream (rows
  // stream * 32 + token, each tile on an 8-row swizzle boundary), so a chunk
  // is one copy each instead of four (the SM's TMA issue rate bounds the
  // chunk rate at small T)
  const cuuint64_t d3[3] = {(cuuint64_t)H, T, 4};
  const cuuint64_t s3[2] = {(cuuint64_t)H * 8, (cuuint64_t)H * 2};
  const cuuint32_t b3[3] = {kChunk, kBM, 4};
  const cuuint64_t d2[2] = {(cuuint64_t)H, T};
  const cuuint64_t s2[1] = {(cuuint64_t)H * 2};
  const cuuint32_t b2[2] = {kChunk, kBM};
  const cuuint64_t dF[3] = {(cuuint64_t)H, kFnRows, 4};
  const cuuint32_t bF[3] = {kChunk, kFnRows, 4};
  const cuuint64_t sC[1] = {(cuuint64_t)H};
  bool ok = encode(&mR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.R, d3, s3, b3, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode(&mRo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.res_out ? (const void*)a.res_out : (const void*)a.R, d3, s3,
                   b3, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode(&mFn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.fn_packed, dF, s3, bF, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode(&mN, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.norm ? (const void*)a.norm : (const void*)a.R, d2, s2, b2,
                   CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok) ok = encode(&mY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.Y ? (const void*)a.Y : (const void*)a.R, d2, s2, b2,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (ok) {  // the quantised output: e4m3 codes (u8), or the fp8_grid (bf16, laid out like the norm)
    if (a.grid)
      ok = encode(&mC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.grid, d2, s2, b2, CU_TENSOR_MAP_SWIZZLE_128B);
    else
      ok = encode(&mC, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.codes ? (const void*)a.codes : (const void*)a.norm, d2, sC,
                  b2, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  // carried gates: comb [T, 16], pre and post [T, 4] fp32, 32 token rows per box
  CUtensorMap mGc, mGp, mGq;
  const cuuint64_t dG16[2] = {16, T}, sG16[1] = {64}, dG4[2] = {4, T}, sG4[1] = {16};
  const cuuint32_t bG16[2] = {16, kBM}, bG4[2] = {4, kBM};
  if (ok) ok = encode(&mGp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.pre_prev, dG4, sG4, bG4, CU_TENSOR_MAP_SWIZZLE_NONE) &&
               encode(&mGq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.post_prev ? a.post_prev : a.pre_prev, dG4, sG4, bG4,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  // the identity form loads no comb: its map slot holds the pre map, never used
  if (ok && a.comb_prev)
    ok = encode(&mGc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.comb_prev, dG16, sG16, bG16, CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    mGc = mGp;
  if (!ok) return cudaErrorInvalidValue;
  MapSet& c = cache[cache_next];
  cache_next = (cache_next + 1) % 4;
  c.T = a.T;
  c.H = H;
  c.out = out_mode;
  for (int i = 0; i < 9; ++i) c.key[i] = key[i];
  c.m[0] = mR; c.m[1] = mY; c.m[2] = mRo; c.m[3] = mFn; c.m[4] = mN; c.m[5] = mC; c.m[6] = mGc; c.m[7] = mGp;
  c.m[8] = mGq;
  return launch_with_maps(a, c.m, tcgen05_proj, kcl, stream, report_ns, launches, wsx, wave_split);
}

// One seam call, one launch.  (Running a partial last round as a second
// launch over larger clusters was measured slower than the partial round; the
// column split of that round runs inside the one launch.)
static cudaError_t launch_with_maps(const SeamArgs& a, const CUtensorMap* m, bool tcgen05_proj, int kcl,
                                    cudaStream_t stream, unsigned long long report_ns, int* launches, void* wsx,
                                    int wave_split) {
  const int n_blocks = (int)((a.T + kBM - 1) / kBM);
  return launch_range(a, m, tcgen05_proj, kcl, 0, n_blocks, stream, report_ns, launches, wsx, wave_split);
}

static cudaError_t launch_range(const SeamArgs& a, const CUtensorMap* m, bool tcgen05_proj, int kcl, int block0,
                                int n_blocks, cudaStream_t stream, unsigned long long report_ns, int* launches,
                                void* wsx, int wave_split) {
  const bool ms = !tcgen05_proj;
  unsigned long long abort_ns = report_ns + 1000000000ull;
  const int form = a.comb_prev == nullptr ? 2 : a.Y != nullptr ? 1 : 0;
  const int mx = a.grid ? 2 : a.codes ? 1 : 0;
  const int fit = max_clusters(form, mx, ms, kcl, 0);
  if (fit <= 0) return cudaErrorInvalidValue;
  const int ncl = n_blocks < fit ? n_blocks : fit;
  int parts = wsx ? wave_parts(n_blocks, ncl, a.H / kChunk, kcl, tcgen05_proj, wave_split) : 1;
  // the split variant's clusters must all be resident at once (cooperative launch)
  if (parts > 1 && max_clusters(form, mx, ms, kcl, 2) < ncl) parts = 1;
  // tickets where the variant exists and there is more than one round
  const int sched = parts > 1 ? 2 : (wsx && n_blocks > ncl && stream_kernel_ptr(form, mx, ms, kcl, 1) != nullptr ? 1 : 0);
  void* k = stream_kernel_ptr(form, mx, ms, kcl, sched);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)kcl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // The kernel's set-up may overlap the previous kernel on the stream (it
  // waits for that kernel before touching global memory).
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  // The parts of a split block wait for each other's partial sums: every
  // cluster of the grid must be resident at once, which a cooperative launch
  // guarantees (the grid is at most the clusters that fit).  Taking tickets
  // needs no co-residency: a cluster that starts late takes what is left.
  attr[2].id = cudaLaunchAttributeCooperative;
  attr[2].val.cooperative = 1;
  cfg.gridDim = dim3((unsigned)(ncl * kcl), 1, 1);
  cfg.blockDim = dim3(mx == 2 ? threads_of<2>() : threads_of<0>(), 1, 1);
  cfg.dynamicSmemBytes = smem_bytes(kcl, mx, form, ms);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = parts > 1 ? 3 : 2;
  // tickets: NB whole blocks, then the last R blocks in `parts` column parts
  int b0 = block0, rsplit = parts > 1 ? n_blocks % ncl : 0, nb_whole = n_blocks - rsplit;
  int kpart = rsplit > 0 ? parts : 1, groups = (a.H / kChunk + kcl - 1) / kcl;
  char* w = static_cast<char*>(wsx);
  void* args[] = {const_cast<SeamArgs*>(&a),    const_cast<CUtensorMap*>(m),     const_cast<CUtensorMap*>(m + 1),
                  const_cast<CUtensorMap*>(m + 2), const_cast<CUtensorMap*>(m + 3), const_cast<CUtensorMap*>(m + 4),
                  const_cast<CUtensorMap*>(m + 5), const_cast<CUtensorMap*>(m + 6), const_cast<CUtensorMap*>(m + 7),
                  const_cast<CUtensorMap*>(m + 8), &b0, &nb_whole, &rsplit, &kpart, &groups, &w, &report_ns, &abort_ns};
  cudaError_t e = cudaLaunchKernelExC(&cfg, k, args);
  if (e == cudaSuccess) {
    ++*launches;
    g_last_parts = parts;
  }
  return e;
}

}  // namespace mhc
