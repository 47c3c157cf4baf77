// Weight-streaming GEMM (host side): launch geometry, tensor maps, and the
// Medusa-head and LM-head entry points.  The kernel and its design notes are
// in wgemm_kernel.cuh; its instances are compiled in wgemm_f32.cu,
// wgemm_silu.cu and wgemm_stats.cu.
#include "wgemm_kernel.cuh"

using namespace sv::wg;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D bf16 map (K, d1, d2) with row pitch K and plane pitch d1 * K elements;
// box (64, box1, 1-or-box2), 128-byte swizzle; out-of-range rows read as 0.
int map3(CUtensorMap *m, const void *base, int K, int d1, int d2, int box1, int box2) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SPEC_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)d1, (cuuint64_t)d2};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * 2 * (cuuint64_t)d1};
  const cuuint32_t box[3] = {(cuuint32_t)kKC, (cuuint32_t)box1, (cuuint32_t)box2};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

inline int pick_nt(int rows) { return rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : rows <= 128 ? 128 : 256; }
inline int pick_mt(int nt) { return nt <= 128 ? 2 : 1; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// One GEMM's launch geometry and workspace: the partial slots (two per CTA).
SvGemmPlan sv_wgemm_plan(int M, int K, int G, int rows) {
  SvGemmPlan p{};
  const int rl = rows < 256 ? rows : 256;  // rows per launch
  p.nt = pick_nt(rl);
  p.mt = pick_mt(p.nt);
  const int km = 128 * p.mt;
  p.nk = K / kKC;
  p.tiles_pg = (M + km - 1) / km;
  p.n_tiles = p.tiles_pg * G;
  p.units = (long long)p.n_tiles * p.nk;
  // (no device: sized for a large GPU, so workspace queries stay meaningful;
  // nothing launches without one)
  const int sms = sm_count() > 0 ? sm_count() : 1024;
  p.n_ctas = (int)(p.units < sms ? p.units : sms);
  p.rows_per_launch = rl;
  // the fixup launch runs when some tile is cut
  auto cta_of = [&](long long x) { return ((x + 1) * p.n_ctas - 1) / p.units; };  // the kernel's cta_of_unit
  p.any_cut = false;
  for (long long t = 0; p.units > 0 && t < p.n_tiles && !p.any_cut; ++t)
    p.any_cut = cta_of(t * p.nk) != cta_of(t * p.nk + p.nk - 1);
  p.partial_bytes = align256((size_t)2 * p.n_ctas * ((rl + 3) / 4 * 4) * km * 4);
  return p;
}

namespace {

// Sums the partials of the tiles a deferred launch cut, in CTA order, and
// stores the epilogue's result (the in-kernel reduction's arithmetic, spread
// over the whole GPU: thread = (tile, 4 activation rows, W row)).
template <int EPI>
__global__ void __launch_bounds__(256) wgemm_fixup_kernel(const WArgs a, int kM) {
  grid_dep_wait();  // every contributor's partial is stored
  const Phase &ph = a.ph;
  const int rows4 = (a.rows + 3) >> 2;
  const long long n = (long long)ph.n_tiles * rows4 * kM;
  const float4 *part = reinterpret_cast<const float4 *>(ph.partial);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int mm = (int)(i % kM);
    const long long tq = i / kM;
    const int q = (int)(tq % rows4), t = (int)(tq / rows4);
    const long long tu = (long long)t * a.nk;
    const int c_first = cta_of_unit(tu, ph.units, a.n_ctas);
    const int c_last = cta_of_unit(tu + a.nk - 1, ph.units, a.n_ctas);
    if (c_first == c_last) continue;  // a whole tile: stored by the GEMM itself
    const int slot_first = 2 * c_first + (range_start(c_first, ph.units, a.n_ctas) >= tu ? 0 : 1);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = c_first; c <= c_last; ++c) {
      const int sl = c == c_first ? slot_first : 2 * c;
      const float4 v = __ldcg(part + ((long long)sl * rows4 + q) * kM + mm);
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
    store4<EPI>(a, ph, t / ph.tiles_pg, (t % ph.tiles_pg) * kM + mm, 0, 4 * q, sum);
  }
}

// The statistics epilogue's fixup: one warp per (cut tile, epilogue quarter,
// 4 activation rows), lane = W row within the quarter: the contributors'
// partials are summed in CTA order, each lane merges its MT W rows, and a
// butterfly over the warp leaves one record per row (the union over the
// quarter's 32 * MT W rows).
__global__ void __launch_bounds__(256) wgemm_fixup_stats_kernel(const WArgs a, int mt_n) {
  grid_dep_wait();  // every contributor's partial is stored
  const Phase &ph = a.ph;
  const int kM = 128 * mt_n, rows4 = (a.rows + 3) >> 2;
  const int lane = threadIdx.x & 31;
  const long long n = (long long)ph.n_tiles * 4 * rows4;
  const float4 *part = reinterpret_cast<const float4 *>(ph.partial);
  for (long long wi = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; wi < n;
       wi += ((long long)gridDim.x * blockDim.x) >> 5) {
    const int q = (int)(wi % rows4), quarter = (int)((wi / rows4) & 3), t = (int)(wi / rows4 / 4);
    const long long tu = (long long)t * a.nk;
    const int c_first = cta_of_unit(tu, ph.units, a.n_ctas);
    const int c_last = cta_of_unit(tu + a.nk - 1, ph.units, a.n_ctas);
    if (c_first == c_last) continue;  // a whole tile: its records are the GEMM's own (warp-uniform)
    const int slot_first = 2 * c_first + (range_start(c_first, ph.units, a.n_ctas) >= tu ? 0 : 1);
    const int mt = t % ph.tiles_pg, ml = quarter * 32 + lane;
    St e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = St{-INFINITY, 0.f, 0.f, 0ull};
    for (int j = 0; j < mt_n; ++j) {
      const int m = mt * kM + j * 128 + ml;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = c_first; c <= c_last; ++c) {
        const int sl = c == c_first ? slot_first : 2 * c;
        const float4 v = __ldcg(part + ((long long)sl * rows4 + q) * kM + j * 128 + ml);
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
      }
      const bool vm = m < ph.M;
      e[0] = st_merge(e[0], st_one(sum.x, m, vm, a.inv_t));
      e[1] = st_merge(e[1], st_one(sum.y, m, vm, a.inv_t));
      e[2] = st_merge(e[2], st_one(sum.z, m, vm, a.inv_t));
      e[3] = st_merge(e[3], st_one(sum.w, m, vm, a.inv_t));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
      for (int i = 0; i < 4; ++i) e[i] = st_merge(e[i], st_shfl(e[i], o));
    if (lane < 4 && 4 * q + lane < a.rows) {
      const St r = lane == 0 ? e[0] : lane == 1 ? e[1] : lane == 2 ? e[2] : e[3];
      a.stats[(long long)(a.r0 + 4 * q + lane) * a.rec_stride + mt * 4 + quarter] =
          make_float4(r.k ? sv::key_value(r.k) : 0.f, r.S, r.Q, __int_as_float(r.k ? (int)sv::key_index(r.k) : -1));
    }
  }
}

template <int EPI>
int launch_fixup(const SvGemmPlan &p, const WArgs &a, cudaStream_t stream) {
  const long long n = EPI == kEpiStats ? (long long)p.n_tiles * 4 * ((a.rows + 3) / 4) * 32
                                       : (long long)p.n_tiles * ((a.rows + 3) / 4) * (128 * p.mt);
  const long long blocks = (n + 255) / 256, cap = 8ll * sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks < cap ? blocks : cap));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if constexpr (EPI == kEpiStats) {
    e = cudaLaunchKernelEx(&cfg, wgemm_fixup_stats_kernel, a, p.mt);
  } else {
    e = cudaLaunchKernelEx(&cfg, wgemm_fixup_kernel<EPI>, a, 128 * p.mt);
  }
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

Phase make_phase(const SvGemmPlan &p, int M, int x_grouped, int epi, float *out, void *zout, const void *res,
                 const void *bias, float *partial) {
  Phase ph{};
  ph.M = M;
  ph.tiles_pg = p.tiles_pg;
  ph.n_tiles = p.n_tiles;
  ph.x_grouped = x_grouped;
  ph.epi = epi;
  ph.units = p.units;
  ph.out = out;
  ph.zout = reinterpret_cast<__nv_bfloat16 *>(zout);
  ph.res = reinterpret_cast<const __nv_bfloat16 *>(res);
  ph.bias = reinterpret_cast<const __nv_bfloat16 *>(bias);
  ph.partial = partial;
  return ph;
}

}  // namespace

// One weight-streaming GEMM over all activation rows (one launch, plus its
// fixup when a tile is cut, per block of up to 256 rows).  x: [rows, Gx, K]
// bf16 (Gx = G when x_grouped, else 1).  `pdl`: the first launch may overlap
// the previous kernel on the stream (only its X loads wait for that kernel).
int sv_wgemm(const SvGemmPlan &p, const void *w, const void *x, int x_grouped, int M, int K, int G, int rows,
             int epi, float *out, void *zout, const void *res, const void *bias, float *partial, bool pdl,
             int32_t *status, cudaStream_t stream, float inv_t, void *stats) {
  const int km = 128 * p.mt;
  if (p.n_ctas < 1) return SPEC_ERR_CUDA;
  CUtensorMap maps[2];
  if (map3(&maps[0], w, K, M, G, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[1], x, K, x_grouped ? G : 1, rows, 1, p.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  for (int r0 = 0; r0 < rows; r0 += p.rows_per_launch) {
    WArgs a{};
    a.ph = make_phase(p, M, x_grouped, epi, out, zout, res, bias, partial);
    a.K = K;
    a.G = G;
    a.rows = rows - r0 < p.rows_per_launch ? rows - r0 : p.rows_per_launch;
    a.r0 = r0;
    a.nk = p.nk;
    a.n_ctas = p.n_ctas;
    a.status = status;
    const bool dep = pdl && r0 == 0;
    a.pdl_wait = dep ? 1 : 0;
    a.inv_t = inv_t;
    a.stats = reinterpret_cast<float4 *>(stats);
    a.rec_stride = p.tiles_pg * 4;
    int rc = epi == kEpiF32     ? launch_f32(p, maps, a, dep, stream)
             : epi == kEpiStats ? launch_stats(p, maps, a, dep, stream)
                                : launch_silu(p, maps, a, dep, stream);
    if (rc == SPEC_OK && p.any_cut)
      rc = epi == kEpiF32     ? launch_fixup<kEpiF32>(p, a, stream)
           : epi == kEpiStats ? launch_fixup<kEpiStats>(p, a, stream)
                              : launch_fixup<kEpiSiluRes>(p, a, stream);
    if (rc != SPEC_OK) return rc;
  }
  return sv_launch_status();
}

// Medusa heads: z = h + SiLU(W1 h + b1) (bf16), then logits = W2 z (float32):
// two GEMMs (each with its fixup); the W2 launch is a programmatic dependent,
// so its first ring of weight loads is in flight while the W1 results are
// completed, and only its z loads wait for them.  (Both in one persistent
// launch, W2 waiting inside it on a count of stored W1 results, measured
// 2-35 % slower at batch 1-64.)  Workspace: each GEMM's partial slots.
namespace {
struct HeadsLayout {
  SvGemmPlan p1, p2;
  size_t pa1, pa2, total;
};
HeadsLayout heads_layout(int batch, int n_heads, int hidden, int vocab) {
  HeadsLayout l{};
  l.p1 = sv_wgemm_plan(hidden, hidden, n_heads, batch);
  l.p2 = sv_wgemm_plan(vocab, hidden, n_heads, batch);
  l.pa1 = 0;
  l.pa2 = l.pa1 + l.p1.partial_bytes;
  l.total = l.pa2 + l.p2.partial_bytes;
  return l;
}
}  // namespace

size_t sv_medusa_heads_ws_bytes(int batch, int n_heads, int hidden, int vocab) {
  return heads_layout(batch, n_heads, hidden, vocab).total;
}

int sv_medusa_heads(const void *h, const void *w1, const void *b1, const void *w2, int batch, int n_heads,
                    int hidden, int vocab, void *z, float *logits, void *ws, int32_t *status, cudaStream_t stream) {
  const HeadsLayout l = heads_layout(batch, n_heads, hidden, vocab);
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  int rc = sv_wgemm(l.p1, w1, h, 0, hidden, hidden, n_heads, batch, kEpiSiluRes, nullptr, z, h, b1,
                    reinterpret_cast<float *>(base + l.pa1), false, status, stream);
  if (rc != SPEC_OK) return rc;
  return sv_wgemm(l.p2, w2, z, 1, vocab, hidden, n_heads, batch, kEpiF32, logits, nullptr, nullptr, nullptr,
                  reinterpret_cast<float *>(base + l.pa2), true, status, stream);
}

size_t sv_lm_head_ws_bytes(int rows, int hidden, int vocab) {
  return sv_wgemm_plan(vocab, hidden, 1, rows).partial_bytes;
}

int sv_lm_head(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits, void *ws,
               int32_t *status, cudaStream_t stream) {
  const SvGemmPlan p = sv_wgemm_plan(vocab, hidden, 1, rows);
  return sv_wgemm(p, w, hid, 0, vocab, hidden, 1, rows, kEpiF32, logits, nullptr, nullptr, nullptr,
                  reinterpret_cast<float *>(ws), false, status, stream);
}
