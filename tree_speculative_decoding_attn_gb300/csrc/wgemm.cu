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

// One GEMM's launch geometry and workspace: counters (4 per tile) then the
// partial slots (two per CTA).
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
  const int sms = sm_count();
  p.n_ctas = (int)(p.units < sms ? p.units : sms);
  p.rows_per_launch = rl;
  // cut tiles are summed by the fixup launch in single-phase GEMMs (as fast
  // as the last arriving warp or faster at every shape measured, by far
  // when the tiles are few against the CTAs); none cut: no fixup launch
  auto cta_of = [&](long long x) { return ((x + 1) * p.n_ctas - 1) / p.units; };  // the kernel's cta_of_unit
  p.defer = false;
  for (long long t = 0; p.units > 0 && t < p.n_tiles && !p.defer; ++t)
    p.defer = cta_of(t * p.nk) != cta_of(t * p.nk + p.nk - 1);
  p.counter_bytes = align256((size_t)p.n_tiles * 16);
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
  const Phase &ph = a.ph[0];
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
// 16 activation rows), lane = W row within the quarter, as in the kernel:
// the contributors' partials are summed in CTA order, each lane merges its
// MT W rows, and the transpose-reduction leaves one record per row.
__global__ void __launch_bounds__(256) wgemm_fixup_stats_kernel(const WArgs a, int mt_n) {
  grid_dep_wait();  // every contributor's partial is stored
  const Phase &ph = a.ph[0];
  const int kM = 128 * mt_n, rows4 = (a.rows + 3) >> 2, chunks = (a.rows + 15) >> 4;
  const int lane = threadIdx.x & 31;
  const long long n = (long long)ph.n_tiles * 4 * chunks;
  const float4 *part = reinterpret_cast<const float4 *>(ph.partial);
  for (long long wi = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; wi < n;
       wi += ((long long)gridDim.x * blockDim.x) >> 5) {
    const int c0 = (int)(wi % chunks) * 16, quarter = (int)((wi / chunks) & 3), t = (int)(wi / chunks / 4);
    const long long tu = (long long)t * a.nk;
    const int c_first = cta_of_unit(tu, ph.units, a.n_ctas);
    const int c_last = cta_of_unit(tu + a.nk - 1, ph.units, a.n_ctas);
    if (c_first == c_last) continue;  // a whole tile: its records are the GEMM's own (warp-uniform)
    const int slot_first = 2 * c_first + (range_start(c_first, ph.units, a.n_ctas) >= tu ? 0 : 1);
    const int mt = t % ph.tiles_pg, ml = quarter * 32 + lane;
    St e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) e[i] = St{-INFINITY, 0.f, 0.f, 0ull};
    for (int j = 0; j < mt_n; ++j) {
      const int m = mt * kM + j * 128 + ml;
      float4 sum[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = c_first; c <= c_last; ++c) {
        const int sl = c == c_first ? slot_first : 2 * c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = (c0 >> 2) + i;
          if (q >= rows4) break;
          const float4 v = __ldcg(part + ((long long)sl * rows4 + q) * kM + j * 128 + ml);
          sum[i].x += v.x;
          sum[i].y += v.y;
          sum[i].z += v.z;
          sum[i].w += v.w;
        }
      }
      const bool vm = m < ph.M;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        e[4 * i] = st_merge(e[4 * i], st_one(sum[i].x, m, vm, a.inv_t));
        e[4 * i + 1] = st_merge(e[4 * i + 1], st_one(sum[i].y, m, vm, a.inv_t));
        e[4 * i + 2] = st_merge(e[4 * i + 2], st_one(sum[i].z, m, vm, a.inv_t));
        e[4 * i + 3] = st_merge(e[4 * i + 3], st_one(sum[i].w, m, vm, a.inv_t));
      }
    }
    put_record(a, mt * 4 + quarter, c0, st_transpose_reduce16(e));
  }
}

template <int EPI>
int launch_fixup(const SvGemmPlan &p, const WArgs &a, cudaStream_t stream) {
  const long long n = EPI == kEpiStats ? (long long)p.n_tiles * 4 * ((a.rows + 15) / 16) * 32
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
                 const void *bias, int *counters, float *partial) {
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
  ph.counters = counters;
  ph.partial = partial;
  return ph;
}

}  // namespace

// One weight-streaming GEMM over all activation rows (one launch per block of
// up to 256 rows).  x: [rows, Gx, K] bf16 (Gx = G when x_grouped, else 1).
// `counters` (p.counter_bytes) must be zero for the first launch when
// `counters_clear`; otherwise they are cleared here, as they are before every
// later row block.  `pdl`: the first launch may overlap the previous kernel
// on the stream (only its X loads wait for that kernel).
int sv_wgemm(const SvGemmPlan &p, const void *w, const void *x, int x_grouped, int M, int K, int G, int rows,
             int epi, float *out, void *zout, const void *res, const void *bias, int *counters, float *partial,
             bool counters_clear, bool pdl, int32_t *status, cudaStream_t stream, float inv_t, void *stats) {
  const int km = 128 * p.mt;
  if (p.n_ctas < 1) return SPEC_ERR_CUDA;
  CUtensorMap maps[4];
  if (map3(&maps[0], w, K, M, G, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[1], x, K, x_grouped ? G : 1, rows, 1, p.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  maps[2] = maps[0];
  maps[3] = maps[1];
  const bool defer = p.defer;
  for (int r0 = 0; r0 < rows; r0 += p.rows_per_launch) {
    if (!defer && (r0 > 0 || !counters_clear))
      if (cudaMemsetAsync(counters, 0, p.counter_bytes, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    WArgs a{};
    a.ph[0] = make_phase(p, M, x_grouped, epi, out, zout, res, bias, counters, partial);
    a.nphase = 1;
    a.K = K;
    a.G = G;
    a.rows = rows - r0 < p.rows_per_launch ? rows - r0 : p.rows_per_launch;
    a.r0 = r0;
    a.nk = p.nk;
    a.n_ctas = p.n_ctas;
    a.status = status;
    const bool dep = pdl && r0 == 0 && counters_clear;
    a.pdl_wait = dep ? 1 : 0;
    a.inv_t = inv_t;
    a.stats = reinterpret_cast<float4 *>(stats);
    a.rec_stride = p.tiles_pg * 4;
    a.defer = defer ? 1 : 0;
    int rc = epi == kEpiF32     ? launch_f32(p, maps, a, dep, stream)
             : epi == kEpiStats ? launch_stats(p, maps, a, dep, stream)
                                : launch_silu(p, maps, a, dep, stream);
    if (rc == SPEC_OK && defer)
      rc = epi == kEpiF32     ? launch_fixup<kEpiF32>(p, a, stream)
           : epi == kEpiStats ? launch_fixup<kEpiStats>(p, a, stream)
                              : launch_fixup<kEpiSiluRes>(p, a, stream);
    if (rc != SPEC_OK) return rc;
  }
  return sv_launch_status();
}

// Medusa heads: z = h + SiLU(W1 h + b1) (bf16), then logits = W2 z (float32),
// in one persistent launch per block of up to 256 rows: every CTA streams its
// share of W1, then its share of W2; a CTA's first W2 chunks are in flight
// while the last W1 results are stored, and its first z load waits (bounded)
// until all of them are.  Workspace: both phases' counters and the readiness
// count side by side (one memset clears them), then each phase's partial
// slots.
namespace {
struct HeadsLayout {
  SvGemmPlan p1, p2;
  size_t c1, c2, ready, pa1, pa2, total;
};
HeadsLayout heads_layout(int batch, int n_heads, int hidden, int vocab) {
  HeadsLayout l{};
  l.p1 = sv_wgemm_plan(hidden, hidden, n_heads, batch);
  l.p2 = sv_wgemm_plan(vocab, hidden, n_heads, batch);
  l.c1 = 0;
  l.c2 = l.p1.counter_bytes;
  l.ready = l.c2 + l.p2.counter_bytes;
  l.pa1 = l.ready + 256;
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
  if (l.p1.n_ctas < 1 || l.p2.n_ctas < 1) return SPEC_ERR_CUDA;
  if (l.p1.nt != l.p2.nt) return SPEC_ERR_CUDA;  // same rows: same tile shape
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  if (l.p1.n_ctas != l.p2.n_ctas) {
    // fewer W1 chunks than CTAs: one grid would leave CTAs without W1 work
    // (stream-K assumes none); two launches, the second dependent on the first
    if (cudaMemsetAsync(base, 0, l.ready, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    int rc = sv_wgemm(l.p1, w1, h, 0, hidden, hidden, n_heads, batch, kEpiSiluRes, nullptr, z, h, b1,
                      reinterpret_cast<int *>(base + l.c1), reinterpret_cast<float *>(base + l.pa1), true, false,
                      status, stream);
    if (rc != SPEC_OK) return rc;
    return sv_wgemm(l.p2, w2, z, 1, vocab, hidden, n_heads, batch, kEpiF32, logits, nullptr, nullptr, nullptr,
                    reinterpret_cast<int *>(base + l.c2), reinterpret_cast<float *>(base + l.pa2), true, true, status,
                    stream);
  }
  const int km = 128 * l.p1.mt;
  CUtensorMap maps[4];
  if (map3(&maps[0], w1, hidden, hidden, n_heads, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[1], h, hidden, 1, batch, 1, l.p1.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[2], w2, hidden, vocab, n_heads, km, 1) != SPEC_OK) return SPEC_ERR_CUDA;
  if (map3(&maps[3], z, hidden, n_heads, batch, 1, l.p1.nt) != SPEC_OK) return SPEC_ERR_CUDA;
  const int n_ctas = l.p2.n_ctas;  // both phases are split over the whole grid
  const SvGemmPlan &p = l.p2;
  for (int r0 = 0; r0 < batch; r0 += l.p1.rows_per_launch) {
    if (cudaMemsetAsync(base, 0, l.pa1, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    WArgs a{};
    a.ph[0] = make_phase(l.p1, hidden, 0, kEpiSiluRes, nullptr, z, h, b1, reinterpret_cast<int *>(base + l.c1),
                         reinterpret_cast<float *>(base + l.pa1));
    a.ph[1] = make_phase(l.p2, vocab, 1, kEpiF32, logits, nullptr, nullptr, nullptr,
                         reinterpret_cast<int *>(base + l.c2), reinterpret_cast<float *>(base + l.pa2));
    a.nphase = 2;
    a.K = hidden;
    a.G = n_heads;
    a.rows = batch - r0 < l.p1.rows_per_launch ? batch - r0 : l.p1.rows_per_launch;
    a.r0 = r0;
    a.nk = l.p1.nk;
    a.n_ctas = n_ctas;
    a.status = status;
    a.xready = reinterpret_cast<int *>(base + l.ready);
    a.inv_t = 1.f;
    const int rc = launch_silu_f32(p, maps, a, false, stream);
    if (rc != SPEC_OK) return rc;
  }
  return sv_launch_status();
}

size_t sv_lm_head_ws_bytes(int rows, int hidden, int vocab) {
  const SvGemmPlan p = sv_wgemm_plan(vocab, hidden, 1, rows);
  return p.counter_bytes + p.partial_bytes;
}

int sv_lm_head(const void *hid, const void *w, int rows, int hidden, int vocab, float *logits, void *ws,
               int32_t *status, cudaStream_t stream) {
  const SvGemmPlan p = sv_wgemm_plan(vocab, hidden, 1, rows);
  uint8_t *base = reinterpret_cast<uint8_t *>(ws);
  return sv_wgemm(p, w, hid, 0, vocab, hidden, 1, rows, kEpiF32, logits, nullptr, nullptr, nullptr,
                  reinterpret_cast<int *>(base), reinterpret_cast<float *>(base + p.counter_bytes), false, false,
                  status, stream);
}
