// Host side of the NF4 GEMM: tensor-map encoding, tile-shape choice, launch.
#pragma once
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

struct GemmCall {
  int mode;                          // GEMM_FWD / GEMM_DX
  const __nv_bfloat16* A;            // [M, Kred] bf16, row pitch lda elements
  long long lda;
  const uint8_t* Wp;                 // packed codes [Nw, Kw/2]
  const __nv_bfloat16* ext_a;        // [M, 64] bf16 (when ext_k > 0)
  int force_bn;                      // 0 = choose
  int force_nacc;                    // 0 = choose
  GemmArgs g;
};

template <int NACC, int BN, int S, int SB, int MODE>
static cudaError_t launch_cfg(const GemmCall& c, cudaStream_t st) {
  using C = GemmCfg<NACC, BN, S, SB>;
  auto kern = nf4_gemm_kernel<NACC, BN, S, SB, MODE>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const GemmArgs& g = c.g;
  CUtensorMap tA, tW, tX;
  if (!make_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.A, (uint64_t)g.Kred, (uint64_t)g.M,
                   (uint64_t)c.lda * 2, 64, C::BM, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (MODE == GEMM_FWD) {
    if (!make_map_2d(&tW, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.Wp, (uint64_t)g.Kw / 2, (uint64_t)g.Nw,
                     (uint64_t)g.Kw / 2, 32, C::UNITS, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    if (!make_map_2d(&tW, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.Wp, (uint64_t)g.Kw / 2, (uint64_t)g.Nw,
                     (uint64_t)g.Kw / 2, C::UNITS / 2, 64, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  if (g.ext_k > 0) {
    if (!make_map_2d(&tX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.ext_a, 64, (uint64_t)g.M, 128, 64, C::BM,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    tX = tA;
  }
  // Tile order: consecutive CTAs (one wave) share the operand that is walked slowly.
  // M-fastest keeps each weight tile in L2 for all row tiles; when the activation
  // operand is the larger one (long reductions, e.g. the 32B down-projection's dX) the
  // N-fastest order lets a wave share activation tiles instead.
  GemmArgs ga = g;
  ga.n_fast = (double)g.M * g.Kred * 2.0 > (double)g.Nw * g.Kw * 0.5625;
  const unsigned tm = (unsigned)((g.M + C::BM - 1) / C::BM), tn = (unsigned)((g.Nout + BN - 1) / BN);
  dim3 grid = ga.n_fast ? dim3(tn, tm) : dim3(tm, tn);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(tA, tW, tX, ga);
  return cudaGetLastError();
}

// Pick the tile shape.  Each CTA dequantises its BN x 64 weight tile once per k-step,
// so above 128 rows two accumulators (BM = 256) always pay: they halve the dequant work
// per MMA FLOP (measured 1.4-1.5x faster at every 8B-shape product).  Between BN = 128
// and 256 the tile with the lower (waves x per-CTA time) wins.  Per-CTA time relative
// to BN = 256, measured on the 8B shapes: forward (register-table dequant, one thread
// per row, BN = 128 tiles alternate k-steps between two halves of the dequant warps)
// 0.76; input gradient (shared-memory table dequant) 0.5.  Ties go to BN = 256 for the
// forward and to BN = 128 for the input gradient (measured).
static void choose_tile(int mode, int M, int Nout, int& nacc, int& bn) {
  const int sms = 148;
  if (M > 128) {
    nacc = 2;
    const long long mt = (M + 255) / 256;
    const long long w256 = (mt * ((Nout + 255) / 256) + sms - 1) / sms;
    const long long w128 = (mt * ((Nout + 127) / 128) + sms - 1) / sms;
    const double t128 = mode == GEMM_FWD ? 0.76 : 0.5;
    const double c128 = (double)w128 * t128, c256 = (double)w256;
    bn = (mode == GEMM_FWD ? c128 < c256 - 1e-9 : c128 <= c256 + 1e-9) ? 128 : 256;
    return;
  }
  struct Opt { int nacc, bn, per_sm; } opts[4] = {{2, 256, 1}, {2, 128, 1}, {1, 256, 1}, {1, 128, 2}};
  double best = 1e30;
  for (auto& o : opts) {
    if (o.nacc == 2 && M <= 128) continue;
    long long ctas = (long long)((M + 128 * o.nacc - 1) / (128 * o.nacc)) * ((Nout + o.bn - 1) / o.bn);
    long long waves = (ctas + (long long)sms * o.per_sm - 1) / ((long long)sms * o.per_sm);
    // per-CTA time ~ tile area; two CTAs per SM share it
    double t = (double)waves * (128.0 * o.nacc * o.bn) / o.per_sm;
    // dequant cost per CTA does not shrink with NACC: penalise single-accumulator tiles a little
    if (o.nacc == 1) t *= 1.15;
    if (t < best - 1e-9) { best = t; nacc = o.nacc; bn = o.bn; }
  }
}

static cudaError_t launch_nf4_gemm(const GemmCall& c, cudaStream_t st) {
  const GemmArgs& g = c.g;
  int nacc = 0, bn = 0;
  choose_tile(c.mode, g.M, g.Nout, nacc, bn);
  if (c.force_bn) bn = c.force_bn;
  if (c.force_nacc) nacc = c.force_nacc;
  if (c.mode == GEMM_FWD) {
    if (nacc == 2 && bn == 256) return launch_cfg<2, 256, 3, 2, GEMM_FWD>(c, st);
    if (nacc == 2 && bn == 128) return launch_cfg<2, 128, 4, 2, GEMM_FWD>(c, st);
    if (nacc == 1 && bn == 256) return launch_cfg<1, 256, 4, 2, GEMM_FWD>(c, st);
    return launch_cfg<1, 128, 3, 2, GEMM_FWD>(c, st);
  } else {
    if (nacc == 2 && bn == 256) return launch_cfg<2, 256, 3, 2, GEMM_DX>(c, st);
    if (nacc == 2 && bn == 128) return launch_cfg<2, 128, 4, 2, GEMM_DX>(c, st);
    if (nacc == 1 && bn == 256) return launch_cfg<1, 256, 4, 2, GEMM_DX>(c, st);
    return launch_cfg<1, 128, 3, 2, GEMM_DX>(c, st);
  }
}

}  // namespace ls
