// NF4-dequant-fused bf16 GEMM on the 5th-gen tensor cores (tcgen05 + TMEM).
//
// Frozen base weights of the streamed decoder layers are held as NF4: 4-bit codes
// into the 16-value NormalFloat table, one fp32 absmax per 64 consecutive weights
// of a row (the format QLoRA published; the Soup pages' "quantization: 4bit # NF4",
// Soup: Fine-Tune an 8B Model on a 4 GB GPU, "The Core Idea: Layer Streaming").
//
//   FWD:  Y[M, N]  = X[M, K]  · deq(W)[N, K]^T   (q/k/v/o/gate/up/down, vocab logits)
//   DX:   dX[M, K] = dY[M, N] · deq(W)[N, K]     (frozen-base backward: input grads only)
//
// plus an optional extra reduction stage of 16/32 columns that carries the LoRA
// up-projection:  Y += [u_q | u_v] · B_ext^T  (forward) or  dX += [s du_q | s du_v] · A_ext
// (backward).  deq(w) = bf16_rne(fp32(q[code]) * absmax): one fp32 multiply and one
// rounding, identical bit for bit to the host definition.
//
// Pipeline per CTA (BM x BN output tiles, BM = 128 x NACC, one after another as the
// tile schedule GemmSched hands them out: whole tiles, or k-ranges of split tiles):
//   warp 0      TMA producer: activation tile (SW128, K-major) + packed code tile,
//               and the tile's absmax values by cp.async, into an S-deep ring.
//   warps 2..9  dequantise codes into a SW128 bf16 tile, an SB-deep ring (one thread
//               per 64-code row with register byte tables; K-major for FWD, MN-major
//               -- W's own orientation -- for DX); then run the epilogue.
//   warp 1      one thread issues tcgen05.mma (M=128, N=BN, K=16) into TMEM
//               accumulators, NACC of them sharing each dequantised B tile.
// Epilogues: bf16 store (+ residual), fp32 store / accumulate, vocabulary
// log-sum-exp partials with target-logit capture, and dlogits for the backward.
#pragma once
#include "common.cuh"

namespace ls {

__device__ __constant__ float kNF4Table[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020814657211f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

__device__ float g_zero_word[4] = {0.f, 0.f, 0.f, 0.f};

// The same 16 values as compile-time constants (folded into the multiplies).
__device__ constexpr float kNF4Values[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020814657211f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

enum GemmMode : int { GEMM_FWD = 0, GEMM_DX = 1 };
enum GemmEpi : int { EPI_BF16 = 0, EPI_F32 = 1, EPI_F32_ACC = 2, EPI_LOGPROB = 3, EPI_DLOGITS = 4 };

struct GemmArgs {
  int M, Nout, Kred;                 // output [M, Nout]; reduction length (multiple of 64)
  int Nw, Kw;                        // W is [Nw, Kw]: FWD Nw=Nout, Kw=Kred; DX Nw=Kred, Kw=Nout
  const float* absmax;               // [Nw, Kw/64]
  int ext_k;                         // 0, 16 or 32 extra reduction columns
  const __nv_bfloat16* ext_b;        // [Nout, 64] (columns >= ext_k are zero)
  int epi;
  void* out;
  long long ldo;
  const __nv_bfloat16* residual;     // EPI_BF16: optional [M, Nout] added before rounding
  long long ldr;
  const int* targets;                // EPI_LOGPROB / EPI_DLOGITS: global target id per row, -1 none
  int vocab_off;                     // global id of output column 0
  float* part_max;                   // EPI_LOGPROB: [M, part_ld] partial max / sum-exp
  float* part_sum;
  int part_ld;
  float* tgt_logit;                  // EPI_LOGPROB: [M] logit of the target
  const float* lse;                  // EPI_DLOGITS: [M]
  const float* coef;                 // EPI_DLOGITS: [M] dL/dlogprob per row
  int n_fast;                        // tile order walks output-column tiles first (a wave shares A rows)
  // Tile schedule (see GemmSched): tiles_m x tiles_n output tiles over sched_ctas CTAs.
  int tiles_m, tiles_n;
  int sched_ctas;                    // CTAs of the launch
  int sched_dp;                      // whole tiles per CTA, tile j * sched_ctas + cta, taken first
  long long sk_iters;                // k-iterations of the remaining tiles, split evenly over the CTAs
  float* sk_ws;                      // split tiles: one fp32 partial slot (kSkSlotFloats) per CTA
  unsigned* sk_flags;                // [sched_ctas][8]: epoch word per (CTA, epilogue warp)
  unsigned sk_epoch;                 // this launch's nonzero epoch
  // Split schedule on a paired batch [first half; second half] of 2 * pair_rows rows: the
  // two accumulators of a tile take rows m0 + a * pair_rows, so row r and row pair_rows + r
  // always share a CTA, its k-ranges and its partial sums (identical inputs -> identical
  // outputs).  0: a tile's accumulators take consecutive 128-row blocks.
  int pair_rows;
};

// Stream-K workspace: one 256 x 256 fp32 partial tile per CTA, at most kSkMaxCtas CTAs.
constexpr int kSkMaxCtas = 148;
constexpr int kSkSlotFloats = 256 * 256;

// Work of one CTA as a sequence of pieces (tile, k-iterations [k0, k1)).  First the
// round-robin whole tiles j * G + c (j < sched_dp; with sched_ctas = tiles and
// sched_dp = 1 this is one tile per CTA), then the CTA's contiguous share
// [c I / G, (c+1) I / G) of the I = sk_iters iterations that the remaining tiles span in
// (tile, k) order.  A share that starts inside a tile leaves a partial sum for the CTA
// that holds the tile's k = 0 piece; that CTA adds the partials of the following CTAs
// (the ones whose shares start inside the tile, in increasing order) before its
// epilogue.  Every CTA's share is non-empty (I >= G, checked on the host), so each
// split tile's partials come from the immediately following CTAs.
// SPLIT = false compiles the one-tile-per-CTA form (tile = CTA index, all k) with no
// trace of the split machinery.
template <bool SPLIT>
struct GemmSched {
  int c, G, ndp, niter, tm, tn, nf, j;
  long long I, pos, end;
  __device__ __forceinline__ void init(const GemmArgs& g, int cta, int niter_) {
    c = cta;
    G = g.sched_ctas;
    ndp = g.sched_dp;
    niter = niter_;
    tm = g.tiles_m;
    tn = g.tiles_n;
    nf = g.n_fast;
    I = SPLIT ? g.sk_iters : 0;
    j = 0;
    pos = SPLIT ? start(c) : 0;
    end = SPLIT ? start(c + 1) : 0;
  }
  __device__ __forceinline__ long long start(int d) const { return (long long)d * I / G; }
  // next piece: tile id, k-iteration range; false when the CTA's work is done
  __device__ __forceinline__ bool next(int& tile, int& k0, int& k1) {
    if constexpr (!SPLIT) {
      if (j) return false;
      j = 1;
      tile = c;
      k0 = 0;
      k1 = niter;
      return true;
    }
    if (j < ndp) {
      tile = j * G + c;
      k0 = 0;
      k1 = niter;
      ++j;
      return true;
    }
    if (pos < end) {
      const long long t = pos / niter;
      k0 = (int)(pos - t * niter);
      const long long rem = end - pos;
      k1 = rem < (long long)(niter - k0) ? k0 + (int)rem : niter;
      tile = ndp * G + (int)t;
      pos += k1 - k0;
      return true;
    }
    return false;
  }
  __device__ __forceinline__ void tile_origin(int tile, int bm, int bn, int& m0, int& n0) const {
    if (nf) {
      n0 = (tile % tn) * bn;
      m0 = (tile / tn) * bm;
    } else {
      m0 = (tile % tm) * bm;
      n0 = (tile / tm) * bn;
    }
  }
  // CTAs c+1 .. last whose shares start inside split tile `tile` (its k = 0 piece is c's)
  __device__ __forceinline__ int last_peer(int tile) const {
    const long long tend = (long long)(tile - ndp * G + 1) * niter;
    int d = c + 1;
    while (d + 1 < G && start(d + 1) < tend) ++d;
    return d;
  }
};

// Dequant warps of the 256 x 256 tiles: 16, in two groups taking alternate k-steps, so
// four of them share each scheduler and hide one another's latency (the dequant is the
// kernel's bound: byte permutes and bit-selects on the integer pipe); 8 elsewhere.
#ifndef LS_GEMM_DQ_WARPS_256
#define LS_GEMM_DQ_WARPS_256 16
#endif

template <int NACC, int BN, int S, int SB>
struct GemmCfg {
  static constexpr int BM = 128 * NACC;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int UNITS = BN;               // 64-element rows dequantised per k-step
  static constexpr int W_BYTES = UNITS * 32;
  static constexpr int ABS_PER_STAGE = UNITS;
  static constexpr int NDQ_WARPS = (NACC == 2 && BN == 256) ? LS_GEMM_DQ_WARPS_256 : 8;
  static constexpr int NDQ = NDQ_WARPS * 32;
  // the first 8 dequant warps also run the epilogue (two per TMEM lane quarter)
  static constexpr int EPI_WARPS = 8;
  // dequant: one thread per 64-element row of the B tile (forward: output column;
  // input gradient: W row x 64-column block); when there are fewer rows than dequant
  // threads, groups of them take alternate k-steps (group g owns B buffer g)
  static constexpr int FWD_GROUPS = NDQ / UNITS;
  static constexpr int FWD_GROUP_WARPS = NDQ_WARPS / FWD_GROUPS;
  static constexpr int THREADS = 64 + NDQ;
  static constexpr int TMEM_COLS = NACC * BN;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + S * A_BYTES;
  static constexpr int OFF_W = OFF_B + SB * B_BYTES;
  static constexpr int OFF_ABS = OFF_W + S * W_BYTES;
  static constexpr int OFF_BAR = OFF_ABS + S * ABS_PER_STAGE * 4;
  static constexpr int NBAR = 2 * S + 2 * SB + 3;   // + accumulator full / drained, TMEM free
  static constexpr int OFF_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_SLOT + 16 + 1024;   // + slack to align the base to 1024
  static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM columns");
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(FWD_GROUPS == 1 || (FWD_GROUPS == 2 && SB == 2), "dequant groups need one B buffer each");
  static_assert(NDQ % UNITS == 0 && NDQ_WARPS >= EPI_WARPS, "dequant warp layout");
};

// -------------------------------------------------------------------------- dequantisers

// FWD, register tables: one thread turns one whole B-tile row (64 codes, one absmax a)
// into bf16.  The 16 possible outputs bf16_rne(q[i] * a) are formed once per row (16
// fp32 multiplies, the same single multiply and rounding as above, so the result is
// bit-identical) and split into low-byte / high-byte tables of four registers each;
// every group of four codes is then looked up with byte permutes (prmt): entries 0..7
// and 8..15 separately, chosen per byte by the code's top bit.  No shared-memory load
// sits inside the per-element chain, so the eight dequant warps stay issue-bound
// instead of waiting on table loads.
struct Nf4ByteTab {
  uint32_t lo[4], hi[4];
};

__device__ __forceinline__ void nf4_byte_tab(float a, Nf4ByteTab& t) {
  uint32_t p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = pack_bf16x2(kNF4Values[2 * i] * a, kNF4Values[2 * i + 1] * a);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t.lo[i] = __byte_perm(p[2 * i], p[2 * i + 1], 0x6420);
    t.hi[i] = __byte_perm(p[2 * i], p[2 * i + 1], 0x7531);
  }
}

// Eight codes (one 32-bit word: byte i holds elements 2i (high nibble) and 2i + 1) to
// four bf16x2 words (elements 0,1 / 2,3 / 4,5 / 6,7).  Per half-word (four codes):
//  - four byte permutes pick each code's low and high output byte from the tables of
//    entries 0..7 and 8..15 (selectors = the codes' low three bits);
//  - one sign-replicating byte permute forms the mask of the codes >= 8: each code's
//    bit 3 is the top bit of a byte of w (even elements) or of w << 4 (odd elements),
//    and a selector nibble with bit 3 set copies that top bit over the whole byte;
//  - two bit-selects merge the halves of the tables, two permutes interleave the low
//    and high bytes into bf16 pairs.
__device__ __forceinline__ void nf4_lookup8(uint32_t w, const Nf4ByteTab& t, uint32_t (&o)[4]) {
  const uint32_t u = w << 4;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t s7 = (h ? w >> 16 : w) & 0x7777u;
    const uint32_t la = prmt(t.lo[0], t.lo[1], s7), lb = prmt(t.lo[2], t.lo[3], s7);
    const uint32_t ha = prmt(t.hi[0], t.hi[1], s7), hb = prmt(t.hi[2], t.hi[3], s7);
    // result bytes in nibble order of s7: elements 1, 0, 3, 2 of this half-word
    const uint32_t m = prmt(w, u, h ? 0xBFAEu : 0x9D8Cu);
    const uint32_t L = (la & ~m) | (lb & m), H = (ha & ~m) | (hb & m);
    o[2 * h] = prmt(L, H, 0x4051u);
    o[2 * h + 1] = prmt(L, H, 0x6273u);
  }
}

// One 64-code row: codes at src (32 bytes, 16-byte aligned), one absmax, written as one
// 128-byte row of the swizzled B tile (dst_off, swizzle phase sw).  h0 staggers the
// order of the two 16-byte code reads across neighbouring rows (bank spread).
__device__ __forceinline__ void dequant_row(const uint8_t* src, float a, int h0, uint8_t* Bt, int dst_off, int sw) {
  const uint4 first = *reinterpret_cast<const uint4*>(src + h0 * 16);
  const uint4 second = *reinterpret_cast<const uint4*>(src + (h0 ^ 1) * 16);
  const uint4 w0 = h0 ? second : first, w1 = h0 ? first : second;
  Nf4ByteTab t;
  nf4_byte_tab(a, t);
  const uint32_t cw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t o[4];
    nf4_lookup8(cw[c], t, o);
    *reinterpret_cast<uint4*>(Bt + dst_off + ((c ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// FWD: unit j = B-tile row base_row + j (output column n0 + base_row + j); its codes
// are row j of this CTA's W tile (32 bytes per row), K-major SW128 destination.
__device__ __forceinline__ void dequant_fwd_unit(const uint8_t* Wt, const float* absS, uint8_t* Bt, int j,
                                                 int base_row) {
  const int jb = base_row + j;
  dequant_row(Wt + j * 32, absS[j], (j >> 2) & 1, Bt, jb * 128, jb & 7);
}

// DX, MN-major B tile.  For dX = dY . deq(W) the MMA's reduction runs over W's rows n
// and its output columns are W's columns k, so W's own row-major tile IS the B operand
// in MN-major form: no transpose.  Unit j = (row n = j % 64, local 64-column block
// j / 64) of this CTA's W tile (wbytes per row), one absmax; stored as one 128-byte
// K-row of the canonical MN-major 128B-swizzled layout: atoms of 64 columns x 8 rows
// (1 KB), 8 atoms down the 64 rows (8 KB per 64 columns):
//   offset = kbl*8192 + (n/8)*1024 + (n%8)*128 + chunk,  kbl = base_kb + j / 64.
__device__ __forceinline__ void dequant_dx_unit(const uint8_t* Wt, const float* absS, uint8_t* Bt, int j, int wbytes,
                                                int base_kb) {
  const int n = j & 63, kbl = j >> 6;
  const int cb = wbytes / 32;   // 64-column blocks in the W tile
  dequant_row(Wt + n * wbytes + kbl * 32, absS[n * cb + kbl], (n >> 1) & 1, Bt,
              (base_kb + kbl) * 8192 + (n >> 3) * 1024 + (n & 7) * 128, n & 7);
}

// LoRA extra stage: B_ext rows [row0, row0 + rows) (K-major, 64 wide) into the B tile.
__device__ __forceinline__ void copy_ext_rows(const __nv_bfloat16* ext_b, int n0, int Nout, uint8_t* Bt, int row0,
                                              int rows, int tq, int nthreads) {
  for (int u = tq; u < rows * 8; u += nthreads) {
    const int j = row0 + (u >> 3), c = u & 7;
    const int n = n0 + j;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < Nout) v = *reinterpret_cast<const uint4*>(ext_b + (size_t)n * 64 + c * 8);
    *reinterpret_cast<uint4*>(Bt + j * 128 + ((c ^ (j & 7)) << 4)) = v;
  }
}

// -------------------------------------------------------------------------- epilogue pieces

__device__ __forceinline__ void store_bf16_16(__nv_bfloat16* dst, const float (&f)[16], int nvalid) {
  if (nvalid >= 16) {
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(p[0], p[1], p[2], p[3]);
    d[1] = make_uint4(p[4], p[5], p[6], p[7]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < nvalid) dst[i] = __float2bfloat16_rn(f[i]);
  }
}

// -------------------------------------------------------------------------- kernel

template <int NACC, int BN, int S, int SB, int MODE, bool SPLIT>
__global__ void __launch_bounds__(GemmCfg<NACC, BN, S, SB>::THREADS, 1)
    nf4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmX, const GemmArgs g) {
  using C = GemmCfg<NACC, BN, S, SB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = g.Kred / 64;
  const int KBw = g.Kw / 64;
  const int niter = KB + (g.ext_k > 0 ? 1 : 0);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + C::OFF_BAR;
  auto full = [&](int s) { return bar0 + s * 8; };
  auto empty = [&](int s) { return bar0 + (S + s) * 8; };
  auto bfull = [&](int s) { return bar0 + (2 * S + s) * 8; };
  auto bempty = [&](int s) { return bar0 + (2 * S + SB + s) * 8; };
  const uint32_t accfull = bar0 + (2 * S + 2 * SB) * 8;       // one phase per piece
  const uint32_t tmemfree = bar0 + (2 * S + 2 * SB + 1) * 8;  // epilogue done reading TMEM
  const uint32_t drained = bar0 + (2 * S + 2 * SB + 2) * 8;   // every MMA retired

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1 + 32);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(bfull(s), C::FWD_GROUP_WARPS);
      mbar_init(bempty(s), 1);
    }
    mbar_init(accfull, 1);
    mbar_init(tmemfree, C::EPI_WARPS);
    mbar_init(drained, 1);
    fence_barrier_init();
    s_abort = 0;
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmW);
    if (g.ext_k > 0) prefetch_tensormap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(sb + C::OFF_SLOT, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT);

  // Every role walks the same piece sequence; gi counts k-iterations across pieces and
  // drives the ring stages and their phases.
  GemmSched<SPLIT> sc;
  sc.init(g, blockIdx.x, niter);
  int tile, k0, k1;

  // rows of a tile: NACC consecutive 128-row blocks, or (split schedule only) the same
  // 128 rows of each half of a paired batch
  const int pair = SPLIT && NACC == 2 ? g.pair_rows : 0;
  const int tile_rows = pair ? 128 : C::BM;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int gi = 0;
    bool stop = false;
    while (!stop && sc.next(tile, k0, k1)) {
      int m0, n0;
      sc.tile_origin(tile, tile_rows, BN, m0, n0);
      for (int it = k0; it < k1; ++it, ++gi) {
        const int s = gi % S;
        if (s_abort || !mbar_wait(empty(s), ((gi / S) & 1) ^ 1)) {
          s_abort = 1;
          stop = true;
          break;
        }
        const uint32_t a_dst = sb + C::OFF_A + s * C::A_BYTES;
        if (lane == 0) {
          if (it < KB) {
            mbar_arrive_expect_tx(full(s), C::A_BYTES + C::W_BYTES);
            if (pair) {   // two 128-row boxes: this tile's rows of each half
              tma_load_2d(a_dst, &tmA, it * 64, m0, full(s));
              tma_load_2d(a_dst + 16384, &tmA, it * 64, m0 + pair, full(s));
            } else {
              tma_load_2d(a_dst, &tmA, it * 64, m0, full(s));
            }
            const uint32_t w_dst = sb + C::OFF_W + s * C::W_BYTES;
            if (MODE == GEMM_FWD) tma_load_2d(w_dst, &tmW, it * 32, n0, full(s));
            else tma_load_2d(w_dst, &tmW, n0 / 2, it * 64, full(s));
          } else {
            mbar_arrive_expect_tx(full(s), C::A_BYTES);
            if (pair) {
              tma_load_2d(a_dst, &tmX, 0, m0, full(s));
              tma_load_2d(a_dst + 16384, &tmX, 0, m0 + pair, full(s));
            } else {
              tma_load_2d(a_dst, &tmX, 0, m0, full(s));
            }
          }
        }
        if (it < KB) {
          const uint32_t abs_dst = sb + C::OFF_ABS + s * C::ABS_PER_STAGE * 4;
          if (MODE == GEMM_FWD) {
            for (int j = lane; j < C::UNITS; j += 32) {
              const int n = n0 + j;
              const float* src = n < g.Nw ? g.absmax + (size_t)n * KBw + it : g_zero_word;
              cp_async_4(abs_dst + j * 4, src);
            }
          } else {
            constexpr int CB = C::UNITS / 64;
            for (int e = lane; e < 64 * CB; e += 32) {
              const int r = e / CB, c = e % CB;
              const int kb = n0 / 64 + c;
              const float* src = kb < KBw ? g.absmax + (size_t)(it * 64 + r) * KBw + kb : g_zero_word;
              cp_async_4(abs_dst + e * 4, src);
            }
          }
        }
        cp_async_mbar_arrive_noinc(full(s));
      }
    }
    if (s_abort) {
      // let copies already in flight land before the CTA's shared memory goes away
      for (int j = gi - S < 0 ? 0 : gi - S; j < gi; ++j) mbar_wait(full(j % S), (j / S) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(128, BN);
      int gi = 0, pc = 0;
      bool stop = false;
      while (!stop && sc.next(tile, k0, k1)) {
        // the epilogue of the previous piece has read TMEM out
        if (pc > 0 && (s_abort || !mbar_wait(tmemfree, (pc - 1) & 1))) {
          s_abort = 1;
          break;
        }
        for (int it = k0; it < k1; ++it, ++gi) {
          const int s = gi % S, b = gi % SB;
          if (s_abort || !mbar_wait(full(s), (gi / S) & 1) || !mbar_wait(bfull(b), (gi / SB) & 1)) {
            s_abort = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const int nk = it < KB ? 4 : g.ext_k / 16;
          const uint32_t a_base = sb + C::OFF_A + s * C::A_BYTES;
          const uint32_t b_base = sb + C::OFF_B + b * C::B_BYTES;
          // the input-gradient main loop reads B MN-major (16 reduction rows = two 1 KB
          // 8-row groups per instruction); the LoRA extra stage is K-major in both modes
          const bool mn = MODE == GEMM_DX && it < KB;
          const uint32_t idesc = mn ? IDESC | (1u << 16) : IDESC;
          for (int k = 0; k < nk; ++k) {
            const uint64_t bd = mn ? sw128_mnmajor_desc(b_base + k * 2048, 8192) : sw128_kmajor_desc(b_base + k * 32);
#pragma unroll
            for (int a = 0; a < NACC; ++a) {
              const uint64_t ad = sw128_kmajor_desc(a_base + a * 16384 + k * 32);
              tc_mma_bf16(tmem + a * BN, ad, bd, idesc, (it > k0 || k > 0) ? 1u : 0u);
            }
          }
          tc_commit(empty(s));
          tc_commit(bempty(b));
        }
        if (stop) break;
        tc_commit(accfull);
        ++pc;
      }
      tc_commit(drained);
      mbar_wait(drained, 0);   // every MMA has retired before TMEM is released
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ dequant warps
    const int tq = threadIdx.x - 64;
    // group grp takes the k-iterations gi = grp (mod FWD_GROUPS); its threads one unit each
    const int grp = tq / C::UNITS;
    const int step = C::FWD_GROUPS;
    const int tg = tq - grp * C::UNITS;
    const int ew = warp - 2;   // epilogue warp: TMEM lane quarter wq, column half `half`
    const int wq = warp & 3;
    const int half = ew >> 2;
    const bool epi = ew < C::EPI_WARPS;
    int gi = 0, pc = 0;
    while (sc.next(tile, k0, k1)) {
      int m0, n0;
      sc.tile_origin(tile, tile_rows, BN, m0, n0);
      const int n = k1 - k0;
      bool stop = false;
      for (int gj = gi + ((grp - gi % step) + step) % step; gj < gi + n; gj += step) {
        const int it = k0 + (gj - gi);
        const int s = gj % S, b = gj % SB;
        if (s_abort || !mbar_wait(full(s), (gj / S) & 1) || !mbar_wait(bempty(b), ((gj / SB) & 1) ^ 1)) {
          s_abort = 1;
          stop = true;
          break;
        }
        uint8_t* Bt = smem + C::OFF_B + b * C::B_BYTES;
        if (it < KB) {
          const uint8_t* Wt = smem + C::OFF_W + s * C::W_BYTES;
          const float* absS = reinterpret_cast<const float*>(smem + C::OFF_ABS + s * C::ABS_PER_STAGE * 4);
          if (MODE == GEMM_FWD) dequant_fwd_unit(Wt, absS, Bt, tg, 0);
          else dequant_dx_unit(Wt, absS, Bt, tg, C::W_BYTES / 64, 0);
        } else {
          copy_ext_rows(g.ext_b, n0, g.Nout, Bt, 0, C::UNITS, tg, C::UNITS);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bfull(b));
      }
      gi += n;
      if (!epi) {   // dequant-only warps go straight on to the next piece's k-steps
        if (stop || s_abort) break;
        continue;
      }
      if (stop || s_abort || !mbar_wait(accfull, pc & 1)) {
        s_abort = 1;
        break;
      }
      tc_fence_after();

      // ---------------------------------------------------------- epilogue of the piece
      // partial: the share started inside the tile -> fp32 partial to this CTA's slot;
      // finish: the tile's k = 0 piece of a split tile -> add the following CTAs' partials.
      // The same (warp, lane) writes and reads each partial element, so a per-warp
      // epoch flag orders them.
      const bool partial = SPLIT && k0 > 0;
      const bool finish = SPLIT && k0 == 0 && k1 < niter;
      const int dlast = finish ? sc.last_peer(tile) : 0;
      if (finish) {
        bool ok = true;
        if (lane == 0)
          for (int d = sc.c + 1; d <= dlast && ok; ++d) ok = flag_wait_eq(g.sk_flags + d * 8 + ew, g.sk_epoch);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        __syncwarp();   // the other lanes' partial loads follow lane 0's acquire
        if (!ok) {
          s_abort = 1;
          break;
        }
      }
      for (int a = 0; a < NACC; ++a) {
        const int row = m0 + a * (pair ? pair : 128) + wq * 32 + lane;
        const bool rok = row < g.M && (!pair || m0 + wq * 32 + lane < pair);
        float run_m = -INFINITY, run_s = 0.f;
        int tgt = -1;
        float lse_r = 0.f, coef_r = 0.f;
        if (!partial && (g.epi == EPI_LOGPROB || g.epi == EPI_DLOGITS)) {
          tgt = rok ? g.targets[row] - g.vocab_off : -1;
          if (g.epi == EPI_DLOGITS && rok) {
            lse_r = g.lse[row];
            coef_r = g.coef[row];
          }
        }
        for (int cc = 0; cc < BN / 32; ++cc) {
          const int c0 = half * (BN / 2) + cc * 16;
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(a * BN + c0), v);
          tmem_ld_wait();
          // partial-slot position of this thread's 16 values: chunk (a, wq, c0 / 16),
          // 4 float4 groups of 32 lanes
          const size_t chunk = ((size_t)(a * 4 + wq) * (BN / 16) + c0 / 16) * 512 + (size_t)lane * 4;
          if (partial) {
            float4* dst = reinterpret_cast<float4*>(g.sk_ws + (size_t)sc.c * kSkSlotFloats + chunk);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              __stcg(dst + q * 32, make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                               __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
            continue;
          }
          const int gc = n0 + c0;
          const int nvalid = min(16, g.Nout - gc);
          if (!rok || nvalid <= 0) continue;
          float f[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
          if (finish) {
            for (int d = sc.c + 1; d <= dlast; ++d) {
              const float4* srcp = reinterpret_cast<const float4*>(g.sk_ws + (size_t)d * kSkSlotFloats + chunk);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 p4 = __ldcg(srcp + q * 32);
                f[4 * q] += p4.x;
                f[4 * q + 1] += p4.y;
                f[4 * q + 2] += p4.z;
                f[4 * q + 3] += p4.w;
              }
            }
          }
          if (g.epi == EPI_BF16) {
            if (g.residual) {
              const __nv_bfloat16* rp = g.residual + (size_t)row * g.ldr + gc;
              if (nvalid >= 16) {
                const uint4* r4 = reinterpret_cast<const uint4*>(rp);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                  const uint4 rv = r4[q];
                  const uint32_t w4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    f[8 * q + 2 * e] += bf16lo(w4[e]);
                    f[8 * q + 2 * e + 1] += bf16hi(w4[e]);
                  }
                }
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  if (i < nvalid) f[i] += bf2f(rp[i]);
              }
            }
            store_bf16_16(reinterpret_cast<__nv_bfloat16*>(g.out) + (size_t)row * g.ldo + gc, f, nvalid);
          } else if (g.epi == EPI_F32 || g.epi == EPI_F32_ACC) {
            float* op = reinterpret_cast<float*>(g.out) + (size_t)row * g.ldo + gc;
            if (nvalid >= 16) {
              float4* o4 = reinterpret_cast<float4*>(op);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float4 x = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
                if (g.epi == EPI_F32_ACC) {
                  const float4 y = o4[q];
                  x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
                }
                o4[q] = x;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (i < nvalid) op[i] = (g.epi == EPI_F32_ACC ? op[i] : 0.f) + f[i];
            }
          } else if (g.epi == EPI_LOGPROB) {
            float cm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (i < nvalid) cm = fmaxf(cm, f[i]);
            if (cm > run_m) {
              run_s *= __expf(run_m - cm);
              run_m = cm;
            }
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (i < nvalid) acc += __expf(f[i] - run_m);
            run_s += acc;
            const int rel = tgt - gc;
            if (rel >= 0 && rel < nvalid) {
              float t = 0.f;
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (i == rel) t = f[i];
              g.tgt_logit[row] = t;
            }
          } else {  // EPI_DLOGITS: coef * (onehot(target) - softmax)
            const int rel = tgt - gc;
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = coef_r * ((i == rel ? 1.f : 0.f) - __expf(f[i] - lse_r));
            store_bf16_16(reinterpret_cast<__nv_bfloat16*>(g.out) + (size_t)row * g.ldo + gc, f, nvalid);
          }
        }
        if (!partial && g.epi == EPI_LOGPROB && rok && n0 + half * (BN / 2) < g.Nout) {
          const int p = (g.vocab_off + n0 + half * (BN / 2)) / (BN / 2);
          g.part_max[(size_t)row * g.part_ld + p] = run_m;
          g.part_sum[(size_t)row * g.part_ld + p] = run_s;
        }
      }
      if (partial) {
        // publish this warp's part of the partial tile
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          st_release_gpu(g.sk_flags + sc.c * 8 + ew, g.sk_epoch);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmemfree);
      ++pc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace ls
