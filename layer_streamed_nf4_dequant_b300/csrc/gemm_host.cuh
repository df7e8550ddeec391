// Host side of the NF4 GEMM: tensor-map encoding, tile-shape choice, launch.
#pragma once
#include <atomic>
#include <mutex>
#include "nf4_gemm.cuh"

namespace ls {

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled get_encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  });
  return fn;
}

// Raise a kernel's dynamic shared-memory limit on the current device, once per device and
// kernel (`done` holds one bit per device; the caller keeps one per kernel).  Concurrent
// first calls both set the same attribute, which is harmless.  Returns the first error.
template <class Kern>
static cudaError_t ensure_smem_attr(Kern kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// 2-D tensor map over a row-major matrix [rows, cols] with row pitch `pitch_bytes`.
static bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                        uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  PFN_encodeTiled enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Stream-K scratch: kSkMaxCtas x 8 epoch words, then one fp32 partial tile per CTA.
// The words must not hold a future epoch before first use (zero-fill once); epochs come
// from one process-wide counter, so no reset between launches is needed.
struct SkWorkspace {
  float* ws = nullptr;
  unsigned* flags = nullptr;
  int pair_rows = 0;   // > 0: the product's rows are two halves that must round alike (plan_schedule)
};
constexpr size_t kSkFlagBytes = 8192;
constexpr size_t kSkWorkspaceBytes = kSkFlagBytes + (size_t)kSkMaxCtas * kSkSlotFloats * sizeof(float);
static_assert((size_t)kSkMaxCtas * 8 * sizeof(unsigned) <= kSkFlagBytes, "flag words");

static inline SkWorkspace sk_workspace_at(void* base) {
  SkWorkspace w;
  if (base) {
    w.flags = reinterpret_cast<unsigned*>(base);
    w.ws = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(base) + kSkFlagBytes);
  }
  return w;
}

static unsigned next_sk_epoch() {
  static std::atomic<unsigned> epoch{0};
  unsigned e = ++epoch;
  if (e == 0) e = ++epoch;
  return e;
}

// CTAs of a split schedule: one per SM (the split tiles use one CTA per SM), at most
// kSkMaxCtas.
static int sk_max_ctas() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kSkMaxCtas;
  static std::atomic<int> cached[64];   // zero-initialised: not yet queried
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = kSkMaxCtas;
    v = sms < kSkMaxCtas ? sms : kSkMaxCtas;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

struct GemmCall {
  int mode;                          // GEMM_FWD / GEMM_DX
  const __nv_bfloat16* A;            // [M, Kred] bf16, row pitch lda elements
  long long lda;
  const uint8_t* Wp;                 // packed codes [Nw, Kw/2]
  const __nv_bfloat16* ext_a;        // [M, 64] bf16 (when ext_k > 0)
  int force_bn;                      // 0 = choose
  int force_nacc;                    // 0 = choose
  SkWorkspace sk;                    // stream-K scratch (none: whole tiles only)
  int split;                         // 0 = by the cost model, 1 = split schedule when possible, -1 = never
  GemmArgs g;
};

// Tile shape and schedule of one product, decided on the host (plan_tile, plan_schedule).
struct GemmPlan {
  int nacc = 0, bn = 0;          // accumulators (tile rows / 128) and tile columns
  bool split = false;            // split schedule wanted (only with NACC = 2 and scratch)
  int tiles_m = 0, tiles_n = 0;  // output tile grid
  int ctas = 0;                  // CTAs launched
  int whole_per_cta = 1;         // round-robin whole tiles per CTA
  long long split_iters = 0;     // k-iterations split evenly over the CTAs (0: none)
  int pair_rows = 0;             // split tiles pair row r with row pair_rows + r (0: no)
};

template <int NACC, int BN, int S, int SB, int MODE>
static cudaError_t launch_cfg(const GemmCall& c, const GemmPlan& p, cudaStream_t st) {
  using C = GemmCfg<NACC, BN, S, SB>;
  // split schedules only for the one-CTA-per-SM (NACC = 2) tiles
  constexpr bool kCanSplit = NACC == 2;
  auto kern_whole = nf4_gemm_kernel<NACC, BN, S, SB, MODE, false>;
  auto kern_split = nf4_gemm_kernel<NACC, BN, S, SB, MODE, kCanSplit>;
  static std::atomic<uint64_t> attr_whole{0}, attr_split{0};
  {
    cudaError_t e = ensure_smem_attr(kern_whole, C::SMEM, attr_whole);
    if (e == cudaSuccess && kCanSplit) e = ensure_smem_attr(kern_split, C::SMEM, attr_split);
    if (e != cudaSuccess) return e;
  }
  const GemmArgs& g = c.g;
  CUtensorMap tA, tW, tX;
  if (!kCanSplit && p.pair_rows) return cudaErrorInvalidValue;
  // a paired tile loads two 128-row boxes (one from each half) per stage
  const uint32_t a_box_rows = p.pair_rows ? 128u : (uint32_t)C::BM;
  if (!make_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.A, (uint64_t)g.Kred, (uint64_t)g.M,
                   (uint64_t)c.lda * 2, 64, a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (MODE == GEMM_FWD) {
    if (!make_map_2d(&tW, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.Wp, (uint64_t)g.Kw / 2, (uint64_t)g.Nw,
                     (uint64_t)g.Kw / 2, 32, C::UNITS, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    if (!make_map_2d(&tW, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.Wp, (uint64_t)g.Kw / 2, (uint64_t)g.Nw,
                     (uint64_t)g.Kw / 2, C::UNITS / 2, 64,
                     C::DX_W_SWIZZLE ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  if (g.ext_k > 0) {
    if (!make_map_2d(&tX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.ext_a, 64, (uint64_t)g.M, 128, 64, a_box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    tX = tA;
  }
  // absmax [Nw, Kw / 64] fp32 by TMA when its row pitch is a multiple of 16 bytes (and, for
  // the input gradient, a tile's 4 k-blocks make a 16-byte box row)
  const int KBw = g.Kw / 64;
  const bool abs_tma = KBw % 4 == 0 && (MODE == GEMM_FWD || C::UNITS == 256) &&
                       (reinterpret_cast<uintptr_t>(g.absmax) & 15) == 0;
  CUtensorMap tS = tA;
  if (abs_tma &&
      !make_map_2d(&tS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax, (uint64_t)KBw, (uint64_t)g.Nw, (uint64_t)KBw * 4,
                   MODE == GEMM_FWD ? 4u : (uint32_t)(C::UNITS / 64), MODE == GEMM_FWD ? (uint32_t)C::UNITS : 64u,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  // bf16 outputs with no residual leave through a tensor map (32-row x 64-column boxes)
  CUtensorMap tO = tA;
  const bool out_tma = C::NDQ_WARPS == C::EPI_WARPS && g.epi == EPI_BF16 && !g.residual && g.M > 0 && g.Nout > 0 && g.ldo % 8 == 0 &&
                       (reinterpret_cast<uintptr_t>(g.out) & 15) == 0 &&
                       make_map_2d(&tO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.out, (uint64_t)g.Nout, (uint64_t)g.M,
                                   (uint64_t)g.ldo * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!out_tma) tO = tA;
  // Tile order: consecutive CTAs (one wave) share the operand that is walked slowly.
  // M-fastest keeps each weight tile in L2 for all row tiles; when the activation
  // operand is the larger one (long reductions, e.g. the 32B down-projection's dX) the
  // N-fastest order lets a wave share activation tiles instead.
  GemmArgs ga = g;
  ga.out_tma = out_tma ? 1 : 0;
  ga.n_fast = (double)g.M * g.Kred * 2.0 > (double)g.Nw * g.Kw * 0.5625;
  const long long nt = (long long)p.tiles_m * p.tiles_n;
  ga.tiles_m = p.tiles_m;
  ga.tiles_n = p.tiles_n;
  ga.sched_ctas = p.ctas;
  ga.sched_dp = p.whole_per_cta;
  ga.pair_rows = p.pair_rows;
  ga.abs_tma = abs_tma ? 1 : 0;
  ga.sk_iters = 0;
  ga.sk_ws = nullptr;
  ga.sk_flags = nullptr;
  ga.sk_epoch = 0;
  if (p.split_iters > 0) {
    if (!kCanSplit || !c.sk.ws || !c.sk.flags) return cudaErrorInvalidValue;
    ga.sk_iters = p.split_iters;
    ga.sk_ws = c.sk.ws;
    ga.sk_flags = c.sk.flags;
    ga.sk_epoch = next_sk_epoch();
  }
  if (!kCanSplit && (ga.sched_dp != 1 || ga.sched_ctas != nt)) return cudaErrorInvalidValue;
  if (ga.sk_iters == 0) {
    if (ga.sched_dp == 1 && ga.sched_ctas == nt && !p.pair_rows)
      kern_whole<<<(unsigned)nt, C::THREADS, C::SMEM, st>>>(tA, tW, tX, tS, tO, ga);
    else   // whole tiles, several per CTA, or paired rows
      kern_split<<<(unsigned)ga.sched_ctas, C::THREADS, C::SMEM, st>>>(tA, tW, tX, tS, tO, ga);
    return cudaGetLastError();
  }
  // CTAs of a split schedule wait for one another's partial tiles: a cooperative launch
  // guarantees they are all resident at once (or fails instead of starting).
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)ga.sched_ctas);
  lc.blockDim = dim3(C::THREADS);
  lc.dynamicSmemBytes = C::SMEM;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kern_split, tA, tW, tX, tS, tO, ga);
}

// Pick the tile shape by estimated time = waves x per-CTA time.  Per-CTA time per
// k-step relative to the 256 x 256 tile, measured on the 3B / 8B / 32B product shapes
// (bench.py --gemm): forward 128x256 (NACC 2, BN 128) 0.76, 128-row tiles BN 256 0.92,
// BN 128 0.62; input gradient 0.67 / 0.87 / 0.60.  128 x 128 tiles fit two CTAs per SM,
// so past one CTA per SM they share it (time x 2 per 296 CTAs).  Grids smaller than the
// SM count finish in one CTA time: there the smallest tile wins (the 3B-shape products
// at 512 rows gain 15-20%); large grids prefer 256 x 256 (half the dequant per MMA FLOP).
static double choose_tile(int mode, int M, int Nout, int& nacc, int& bn) {
  const int sms = 148;
  struct Opt {
    int nacc, bn, per_sm;
    double cost_fwd, cost_dx;
  };
  // in preference order for ties: forward larger tiles first, input gradient (2, 128) first
  const Opt fwd_opts[4] = {{2, 256, 1, 1.0, 1.0}, {2, 128, 1, 0.76, 0.67}, {1, 256, 1, 0.92, 0.87},
                           {1, 128, 2, 0.62, 0.60}};
  const Opt dx_opts[4] = {fwd_opts[1], fwd_opts[0], fwd_opts[2], fwd_opts[3]};
  const Opt* opts = mode == GEMM_FWD ? fwd_opts : dx_opts;
  double best = 1e30;
  for (int i = 0; i < 4; ++i) {
    const Opt& o = opts[i];
    if (o.nacc == 2 && M <= 128) continue;
    const long long ctas = (long long)((M + 128 * o.nacc - 1) / (128 * o.nacc)) * ((Nout + o.bn - 1) / o.bn);
    const double cost = mode == GEMM_FWD ? o.cost_fwd : o.cost_dx;
    const double t = ctas <= sms ? cost
                                 : (double)((ctas + (long long)sms * o.per_sm - 1) / ((long long)sms * o.per_sm)) *
                                       cost * o.per_sm;
    if (t < best - 1e-9) {
      best = t;
      nacc = o.nacc;
      bn = o.bn;
    }
  }
  return best;
}

// With stream-K scratch the 256 x 256 tile can also run as a split schedule: every SM
// gets the same number of k-iterations, so the estimate is tiles / SMs tile times (plus
// the partial-tile exchange) instead of whole waves.  split_pref: 0 = estimate,
// 1 = split whenever possible, -1 = whole tiles.
static void plan_tile(int mode, int M, int Nout, int Kred, int ext_k, bool has_ws, int split_pref, int force_bn,
                      int force_nacc, int sms, GemmPlan& p) {
  const double t_whole = choose_tile(mode, M, Nout, p.nacc, p.bn);
  p.split = false;
  if (has_ws && split_pref >= 0 && M > 128) {
    const double nt = (double)((M + 255) / 256) * (double)((Nout + 255) / 256);
    // the split kernel's k-iteration costs 1.09 x the whole-tile kernel's (measured on
    // the 8B product shapes), plus about 12 k-iterations per CTA for the partial-tile
    // exchange and the extra pipeline fill
    const int niter = Kred / 64 + (ext_k > 0 ? 1 : 0);
    const double t_split = 1.09 * nt / sms + 12.0 / niter;
    if (split_pref > 0 || t_split < t_whole) {
      p.split = true;
      p.nacc = 2;
      p.bn = 256;
    }
  }
  if (force_bn) p.bn = force_bn;
  if (force_nacc) p.nacc = force_nacc;
  if (p.nacc != 2) p.split = false;   // split schedules use one CTA per SM
}

// Whole tiles, one per CTA; or, for a split plan, one CTA per SM (at most `sms`): full
// rounds of whole tiles, then the last one to two rounds' worth of tiles split evenly by
// k-iterations (each CTA at least 4 of them).
// pair_rows > 0 marks a batch of two halves [rows 0..pair_rows); the same rows again] that
// must give identical outputs for identical rows (the shared-read DPO forward: policy and
// reference copies).  Whole tiles do that as they are (every row is summed in k order);
// a split plan pairs the halves instead, its two 128-row accumulators taking row r and
// row pair_rows + r, so both meet the same k-splits.  Without two accumulators, or when
// M is not 2 * pair_rows, the plan falls back to whole tiles.
static void plan_schedule(int M, int Nout, int Kred, int ext_k, int sms, int pair_rows, GemmPlan& p) {
  p.pair_rows = 0;
  if (pair_rows > 0) {
    if (p.split && p.nacc == 2 && M == 2 * pair_rows) p.pair_rows = pair_rows;
    else p.split = false;
  }
  const long long rows = p.pair_rows ? p.pair_rows : M, tile_rows = p.pair_rows ? 128 : 128 * p.nacc;
  const long long tm = (rows + tile_rows - 1) / tile_rows, tn = (Nout + p.bn - 1) / p.bn, nt = tm * tn;
  const int niter = Kred / 64 + (ext_k > 0 ? 1 : 0);
  p.tiles_m = (int)tm;
  p.tiles_n = (int)tn;
  p.ctas = (int)nt;
  p.whole_per_cta = 1;
  p.split_iters = 0;
  if (!p.split) return;
  const long long full = nt / sms;
  if (nt % sms == 0) {
    p.ctas = sms;
    p.whole_per_cta = (int)full;
    return;
  }
  const long long dp = full > 0 ? full - 1 : 0;
  const long long iters = (nt - dp * sms) * niter;
  long long G = sms;
  if (dp == 0 && iters / 4 < G) G = iters / 4 > 0 ? iters / 4 : 1;
  if (G > 1) {
    p.ctas = (int)G;
    p.whole_per_cta = (int)dp;
    p.split_iters = iters;
  }
}

static GemmPlan plan_gemm(const GemmCall& c, int sms) {
  const GemmArgs& g = c.g;
  GemmPlan p;
  plan_tile(c.mode, g.M, g.Nout, g.Kred, g.ext_k, c.sk.ws && c.sk.flags, c.split, c.force_bn, c.force_nacc, sms, p);
  plan_schedule(g.M, g.Nout, g.Kred, g.ext_k, sms, c.sk.pair_rows, p);
  return p;
}

static cudaError_t launch_nf4_gemm(const GemmCall& c, cudaStream_t st) {
  const GemmPlan p = plan_gemm(c, sk_max_ctas());
  if (c.mode == GEMM_FWD) {
    if (p.nacc == 2 && p.bn == 256) return launch_cfg<2, 256, 3, 2, GEMM_FWD>(c, p, st);
    if (p.nacc == 2 && p.bn == 128) return launch_cfg<2, 128, 4, 2, GEMM_FWD>(c, p, st);
    if (p.nacc == 1 && p.bn == 256) return launch_cfg<1, 256, 4, 2, GEMM_FWD>(c, p, st);
    return launch_cfg<1, 128, 3, 2, GEMM_FWD>(c, p, st);
  } else {
    if (p.nacc == 2 && p.bn == 256) return launch_cfg<2, 256, 3, 2, GEMM_DX>(c, p, st);
    if (p.nacc == 2 && p.bn == 128) return launch_cfg<2, 128, 4, 2, GEMM_DX>(c, p, st);
    if (p.nacc == 1 && p.bn == 256) return launch_cfg<1, 256, 4, 2, GEMM_DX>(c, p, st);
    return launch_cfg<1, 128, 3, 2, GEMM_DX>(c, p, st);
  }
}

}  // namespace ls
