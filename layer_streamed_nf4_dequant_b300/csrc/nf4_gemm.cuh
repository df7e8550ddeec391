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
// Epilogues (TMEM read 32 columns at a time): bf16 store (+ residual; without one, the
// rows are staged in the idle B ring as 128-byte-swizzled boxes and leave by TMA
// tensor stores), fp32 store / accumulate, vocabulary log-sum-exp partials with
// target-logit capture, and dlogits for the backward.
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
  // absmax by TMA (1) or 4-byte cp.async (0).  TMA: forward, a box of 4 consecutive k-blocks x
  // UNITS rows each k-step (column it % 4 used); input gradient, the k-step's 64 rows x 4
  // k-blocks.  Needs the absmax row pitch (K / 64 floats) to be a multiple of 16 bytes.
  int abs_tma;
  // EPI_BF16 without residual: 1 = each epilogue warp stages its rows in its slice of the
  // (then idle) B ring in the 128-byte-swizzled box layout and the output tensor map stores
  // them (32 rows x 64 columns per box); 0 = direct row stores
  int out_tma;
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

// A walk over a CTA's items (k-iterations of its pieces, in order), for roles that run
// ahead of the others (the producer's two rings).
template <bool SPLIT>
struct ItemCursor {
  GemmSched<SPLIT> sc;
  int tile, k1, it, m0, n0, trows, bn;
  __device__ __forceinline__ void init(const GemmArgs& g, int cta, int niter, int tile_rows, int bn_) {
    sc.init(g, cta, niter);
    tile = k1 = it = m0 = n0 = 0;
    trows = tile_rows;
    bn = bn_;
  }
  // advance to the next item; false once the CTA's work is done
  __device__ __forceinline__ bool next() {
    if (it + 1 < k1) {
      ++it;
      return true;
    }
    int k0;
    if (!sc.next(tile, k0, k1)) {
      it = k1 = 0;
      return false;
    }
    it = k0;
    sc.tile_origin(tile, trows, bn, m0, n0);
    return true;
  }
};

// Shared-memory rings of one CTA:
//  - A ring (S stages): the activation tile of a k-step, filled by TMA, released by the
//    MMAs that read it;
//  - W ring (SW stages): the packed codes and absmax of a k-step, filled by TMA and
//    cp.async, released by the dequant warps as soon as they have read them.  The
//    producer keeps it LOOK k-steps ahead of the A ring, so a dequant never waits for an
//    MMA to finish before its codes can be fetched;
//  - B ring (SB stages): dequantised bf16 tiles, written by the dequant warps, released
//    by the MMAs; idle during a tile's epilogue, when it holds the staged output boxes.
// Dequant: TPU threads per 64-code row of the B tile (1: the whole row, 2: 32 codes
// each), in NGRP groups taking alternate k-steps (group g owns B buffer g); the first 8
// dequant warps also run the epilogue (two per TMEM lane quarter).  The 256-wide tiles
// take their layout from LS_GEMM_TPU_256 / LS_GEMM_NGRP_256; the 128-wide ones use two
// threads per row, one group.
#ifndef LS_GEMM_TPU_256
#define LS_GEMM_TPU_256 1
#endif
#ifndef LS_GEMM_NGRP_256
#define LS_GEMM_NGRP_256 1
#endif

template <int NACC, int BN, int S, int SB>
struct GemmCfg {
  static constexpr int BM = 128 * NACC;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int UNITS = BN;               // 64-element rows dequantised per k-step
  static constexpr int W_BYTES = UNITS * 32;
  static constexpr int ABS_PER_STAGE = UNITS * 4;   // floats (forward TMA box: 4 k-blocks per row)
  static constexpr int SW = 5;
  static constexpr int LOOK = 3;                 // W ring lead over the A ring (< SW)
  static constexpr int TPU = BN == 256 ? LS_GEMM_TPU_256 : 2;
  static constexpr int NGRP = BN == 256 ? LS_GEMM_NGRP_256 : 1;
  static constexpr int GROUP_THREADS = TPU * UNITS;
  static constexpr int NDQ = GROUP_THREADS * NGRP;
  static constexpr int NDQ_WARPS = NDQ / 32;
  static constexpr int GROUP_WARPS = NDQ_WARPS / NGRP;
  static constexpr int EPI_WARPS = 8;
  // input gradient: the code tile's rows are 128 bytes at BN = 256; TMA stores them with
  // the 128-byte swizzle so that a row-per-lane read pattern meets no bank conflicts
  static constexpr bool DX_W_SWIZZLE = UNITS == 256;
  static constexpr int THREADS = 64 + NDQ;
  static constexpr int TMEM_COLS = NACC * BN;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + S * A_BYTES;
  static constexpr int OFF_W = OFF_B + SB * B_BYTES;
  static constexpr int OFF_ABS = OFF_W + SW * W_BYTES;
  static constexpr int OFF_BAR = OFF_ABS + SW * ABS_PER_STAGE * 4;
  static constexpr int NBAR = 2 * S + 2 * SW + 2 * SB + 3;   // + accumulator full / drained, TMEM free
  static constexpr int OFF_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_SLOT + 16 + 1024;   // + slack to align the base to 1024
  static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM columns");
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(LOOK < SW && NDQ_WARPS >= EPI_WARPS, "ring / warp layout");
  static_assert((TPU == 1 || TPU == 2) && (NGRP == 1 || (NGRP == 2 && SB == 2)), "dequant layout");
  static_assert(SMEM <= 227 * 1024, "shared memory");
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

// Half a 64-code row: 32 codes at src (16 bytes, 16-byte aligned), the row's absmax,
// written as chunks 4 hf .. 4 hf + 3 of one 128-byte row of the swizzled B tile
// (dst_off, swizzle phase sw).
__device__ __forceinline__ void dequant_half(const uint8_t* src, float a, int hf, uint8_t* Bt, int dst_off, int sw) {
  const uint4 w = *reinterpret_cast<const uint4*>(src);
  Nf4ByteTab t;
  nf4_byte_tab(a, t);
  const uint32_t cw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[4];
    nf4_lookup8(cw[c], t, o);
    *reinterpret_cast<uint4*>(Bt + dst_off + (((4 * hf + c) ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// A whole 64-code row: 32 code bytes as two 16-byte pieces at src0 / src1, one absmax,
// written as the 8 chunks of one 128-byte row of the swizzled B tile.
// swap_read: the pieces are read src1 first (bank spread), still fed in k order.
__device__ __forceinline__ void dequant_full(const uint8_t* src0, const uint8_t* src1, float a, uint8_t* Bt,
                                             int dst_off, int sw, int swap_read) {
  const uint4 r0 = *reinterpret_cast<const uint4*>(swap_read ? src1 : src0);
  const uint4 r1 = *reinterpret_cast<const uint4*>(swap_read ? src0 : src1);
  const uint4 w0 = swap_read ? r1 : r0, w1 = swap_read ? r0 : r1;
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

// FWD, one group thread tg of a k-step.  B-tile row j (output column n0 + j) holds the
// 64 codes of row j of this CTA's W tile (32 bytes), K-major SW128 destination.
//  TPU 1: thread tg takes row j = tg; rows j and j ^ 4 read their two 16-byte pieces in
//         opposite order, so the 8 lanes of a 16-byte access phase meet 8 bank groups;
//  TPU 2: thread tg takes half hf = tg & 1 of row j = tg >> 1 (a warp reads 512
//         contiguous bytes).
// Row j's absmax is absS[j * astride + acol] (a k-block column of the TMA box, or one
// float per row).
template <int TPU>
__device__ __forceinline__ void dequant_fwd_part(const uint8_t* Wt, const float* absS, int astride, int acol,
                                                 uint8_t* Bt, int tg) {
  if constexpr (TPU == 1) {
    const int j = tg, h0 = (j >> 2) & 1;
    const uint8_t* lo = Wt + j * 32;
    const uint8_t* hi = lo + 16;
    dequant_full(lo, hi, absS[j * astride + acol], Bt, j * 128, j & 7, h0);
  } else {
    const int j = tg >> 1, hf = tg & 1;
    dequant_half(Wt + j * 32 + hf * 16, absS[j * astride + acol], hf, Bt, j * 128, j & 7);
  }
}

// DX, MN-major B tile.  For dX = dY . deq(W) the MMA's reduction runs over W's rows n
// and its output columns are W's columns k, so W's own row-major tile IS the B operand
// in MN-major form: no transpose.  The W tile has 64 rows of UNITS / 2 bytes; a unit is
// (row n, 64-column block kbl) with one absmax.  Stored as one 128-byte K-row of the
// canonical MN-major 128B-swizzled layout: atoms of 64 columns x 8 rows (1 KB), 8 atoms
// down the 64 rows (8 KB per 64 columns):
//   offset = kbl*8192 + (n/8)*1024 + (n%8)*128 + chunk.
// UNITS 256: the W tile itself arrived 128B-swizzled (16-byte piece q of row n at
// q ^ (n & 7)), and unit u = (n = u % 64, kbl = u / 64) puts 8 different rows in every
// 8-lane access phase, so reads and writes meet 8 bank groups.  TPU 1: thread tg takes
// unit tg; TPU 2: half hf = tg & 1 of unit tg >> 1.
// UNITS 128 (TPU 2, unswizzled 64-byte rows): thread tg takes piece tg % 4 of row tg / 4,
// a warp reading whole contiguous rows.
template <int UNITS, int TPU>
__device__ __forceinline__ void dequant_dx_part(const uint8_t* Wt, const float* absS, uint8_t* Bt, int tg) {
  constexpr int CB = UNITS / 64, WB = UNITS / 2;
  if constexpr (UNITS == 256) {
    const int u = TPU == 1 ? tg : tg >> 1;
    const int n = u & 63, kbl = u >> 6, sw = n & 7;
    const uint8_t* row = Wt + n * WB;
    const int dst = kbl * 8192 + (n >> 3) * 1024 + sw * 128;
    if constexpr (TPU == 1) {
      dequant_full(row + (((2 * kbl) ^ sw) << 4), row + (((2 * kbl + 1) ^ sw) << 4), absS[n * CB + kbl], Bt, dst, sw,
                   0);
    } else {
      const int hf = tg & 1;
      dequant_half(row + (((2 * kbl + hf) ^ sw) << 4), absS[n * CB + kbl], hf, Bt, dst, sw);
    }
  } else {
    static_assert(TPU == 2, "128-wide input-gradient tiles use two threads per unit");
    constexpr int P = UNITS / 32;
    const int n = tg / P, piece = tg % P, kbl = piece >> 1, hf = piece & 1;
    dequant_half(Wt + n * WB + piece * 16, absS[n * CB + kbl], hf, Bt, kbl * 8192 + (n >> 3) * 1024 + (n & 7) * 128,
                 n & 7);
  }
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
                    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmO, const GemmArgs g) {
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
  constexpr int SW = C::SW;
  auto afull = [&](int s) { return bar0 + s * 8; };
  auto aempty = [&](int s) { return bar0 + (S + s) * 8; };
  auto wfull = [&](int s) { return bar0 + (2 * S + s) * 8; };
  auto wempty = [&](int s) { return bar0 + (2 * S + SW + s) * 8; };
  auto bfull = [&](int s) { return bar0 + (2 * S + 2 * SW + s) * 8; };
  auto bempty = [&](int s) { return bar0 + (2 * S + 2 * SW + SB + s) * 8; };
  constexpr int BAR_END = 2 * S + 2 * SW + 2 * SB;
  const uint32_t accfull = bar0 + BAR_END * 8;         // one phase per piece
  const uint32_t tmemfree = bar0 + (BAR_END + 1) * 8;  // epilogue done reading TMEM
  const uint32_t drained = bar0 + (BAR_END + 2) * 8;   // every MMA retired

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(afull(s), 1);
      mbar_init(aempty(s), 1);
    }
    for (int s = 0; s < SW; ++s) {
      mbar_init(wfull(s), 1 + 32);
      mbar_init(wempty(s), C::GROUP_WARPS);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(bfull(s), C::GROUP_WARPS);
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
    if (g.abs_tma) prefetch_tensormap(&tmS);
  }
  if (warp == 1) {
    tmem_alloc(sb + C::OFF_SLOT, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT);

  // Every role walks the same item sequence (the k-iterations of the CTA's pieces, in
  // order); item counters drive the ring stages and their phases.
  GemmSched<SPLIT> sc;
  sc.init(g, blockIdx.x, niter);
  int tile, k0, k1;

  // rows of a tile: NACC consecutive 128-row blocks, or (split schedule only) the same
  // 128 rows of each half of a paired batch
  const int pair = SPLIT && NACC == 2 ? g.pair_rows : 0;
  const int tile_rows = pair ? 128 : C::BM;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Two cursors over the item sequence: W (codes + absmax) runs LOOK items ahead of A.
    // Waits never depend on an item not yet issued: W item w needs the dequant of item
    // w - SW, which needs A item w - SW - SB + 1 (< the A items issued) for its B buffer.
    ItemCursor<SPLIT> cw, ca;
    cw.init(g, blockIdx.x, niter, tile_rows, BN);
    ca.init(g, blockIdx.x, niter, tile_rows, BN);
    int nw = 0, na = 0;
    auto issue_w = [&]() -> bool {
      const int s = nw % SW, it = cw.it;
      if (s_abort || !mbar_wait(wempty(s), ((nw / SW) & 1) ^ 1)) return false;
      const uint32_t abs_dst = sb + C::OFF_ABS + s * C::ABS_PER_STAGE * 4;
      if (lane == 0) {
        if (it < KB) {
          const int abs_bytes = !g.abs_tma ? 0 : MODE == GEMM_FWD ? C::UNITS * 16 : C::UNITS * 4;
          mbar_arrive_expect_tx(wfull(s), C::W_BYTES + abs_bytes);
          const uint32_t w_dst = sb + C::OFF_W + s * C::W_BYTES;
          if (MODE == GEMM_FWD) tma_load_2d(w_dst, &tmW, it * 32, cw.n0, wfull(s));
          else tma_load_2d(w_dst, &tmW, cw.n0 / 2, it * 64, wfull(s));
          if (g.abs_tma) {
            if (MODE == GEMM_FWD) tma_load_2d(abs_dst, &tmS, it & ~3, cw.n0, wfull(s));
            else tma_load_2d(abs_dst, &tmS, cw.n0 / 64, it * 64, wfull(s));
          }
        } else {
          mbar_arrive(wfull(s));   // the LoRA extra stage reads no codes
        }
      }
      if (it < KB && !g.abs_tma) {
        if (MODE == GEMM_FWD) {
          for (int j = lane; j < C::UNITS; j += 32) {
            const int n = cw.n0 + j;
            const float* src = n < g.Nw ? g.absmax + (size_t)n * KBw + it : g_zero_word;
            cp_async_4(abs_dst + j * 4, src);
          }
        } else {
          constexpr int CB = C::UNITS / 64;
          for (int e = lane; e < 64 * CB; e += 32) {
            const int r = e / CB, c = e % CB;
            const int kb = cw.n0 / 64 + c;
            const float* src = kb < KBw ? g.absmax + (size_t)(it * 64 + r) * KBw + kb : g_zero_word;
            cp_async_4(abs_dst + e * 4, src);
          }
        }
      }
      cp_async_mbar_arrive_noinc(wfull(s));
      ++nw;
      return true;
    };
    auto issue_a = [&]() -> bool {
      const int s = na % S, it = ca.it;
      if (s_abort || !mbar_wait(aempty(s), ((na / S) & 1) ^ 1)) return false;
      if (lane == 0) {
        const uint32_t a_dst = sb + C::OFF_A + s * C::A_BYTES;
        const CUtensorMap* map = it < KB ? &tmA : &tmX;
        const int x = it < KB ? it * 64 : 0;
        mbar_arrive_expect_tx(afull(s), C::A_BYTES);
        if (pair) {   // two 128-row boxes: this tile's rows of each half
          tma_load_2d(a_dst, map, x, ca.m0, afull(s));
          tma_load_2d(a_dst + 16384, map, x, ca.m0 + pair, afull(s));
        } else {
          tma_load_2d(a_dst, map, x, ca.m0, afull(s));
        }
      }
      ++na;
      return true;
    };
    bool ok = true;
    for (int i = 0; ok && i < C::LOOK && cw.next(); ++i) ok = issue_w();
    while (ok) {
      if (cw.next()) ok = issue_w();
      if (!ok || !ca.next()) break;
      ok = issue_a();
    }
    if (!ok) {
      s_abort = 1;
      // let copies already in flight land before the CTA's shared memory goes away
      for (int j = nw - SW < 0 ? 0 : nw - SW; j < nw; ++j) mbar_wait(wfull(j % SW), (j / SW) & 1);
      for (int j = na - S < 0 ? 0 : na - S; j < na; ++j) mbar_wait(afull(j % S), (j / S) & 1);
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
          if (s_abort || !mbar_wait(afull(s), (gi / S) & 1) || !mbar_wait(bfull(b), (gi / SB) & 1)) {
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
          tc_commit(aempty(s));
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
    // group grp takes the items gi = grp (mod NGRP); tg = the thread's index in it
    const int grp = tq / C::GROUP_THREADS, tg = tq % C::GROUP_THREADS;
    const int ew = warp - 2;   // epilogue warp: TMEM lane quarter wq, column half `half`
    const int wq = warp & 3;
    const int half = ew >> 2;
    const bool epi = ew < C::EPI_WARPS;
    // staged output boxes borrow the B ring, which only the epilogue warps write
    const bool kOutTma = C::NDQ_WARPS == C::EPI_WARPS && SB * C::B_BYTES >= C::EPI_WARPS * 32 * BN && g.out_tma;
    int gi = 0, pc = 0;
    while (sc.next(tile, k0, k1)) {
      int m0, n0;
      sc.tile_origin(tile, tile_rows, BN, m0, n0);
      bool stop = false;
      for (int it = k0; it < k1; ++it, ++gi) {
        if (C::NGRP > 1 && gi % C::NGRP != grp) continue;
        const int sw = gi % SW, b = gi % SB;
        if (s_abort || !mbar_wait(wfull(sw), (gi / SW) & 1) || !mbar_wait(bempty(b), ((gi / SB) & 1) ^ 1)) {
          s_abort = 1;
          stop = true;
          break;
        }
        uint8_t* Bt = smem + C::OFF_B + b * C::B_BYTES;
        if (it < KB) {
          const uint8_t* Wt = smem + C::OFF_W + sw * C::W_BYTES;
          const float* absS = reinterpret_cast<const float*>(smem + C::OFF_ABS + sw * C::ABS_PER_STAGE * 4);
          if (MODE == GEMM_FWD) dequant_fwd_part<C::TPU>(Wt, absS, g.abs_tma ? 4 : 1, g.abs_tma ? (it & 3) : 0, Bt, tg);
          else dequant_dx_part<C::UNITS, C::TPU>(Wt, absS, Bt, tg);
        } else {
          copy_ext_rows(g.ext_b, n0, g.Nout, Bt, 0, C::UNITS, tg, C::GROUP_THREADS);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(wempty(sw));
          mbar_arrive(bfull(b));
        }
      }
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
        // the tensor store writes whole 32-row boxes: only where every row of the warp's box
        // belongs to this tile (rows past M are clipped by the map)
        const bool tstore = kOutTma && !partial && (!pair || m0 + wq * 32 + 32 <= pair);
        uint8_t* ostg = smem + C::OFF_B + ew * (32 * BN);   // this warp's 32 x BN / 2 bf16 boxes
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
        for (int cp = 0; cp < BN / 64; ++cp) {
          // 32 columns per TMEM load, and the peers' partials of both 16-column chunks are
          // all in flight before the first is added: the epilogue is latency-bound
          const int cb = half * (BN / 2) + cp * 32;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(a * BN + cb), v);
          tmem_ld_wait();
          // partial-slot position of this thread's values: chunks (a, wq, cb / 16) and the next
          // one (512 floats on), each 4 float4 groups of 32 lanes
          const size_t chunk = ((size_t)(a * 4 + wq) * (BN / 16) + cb / 16) * 512 + (size_t)lane * 4;
          if (partial) {
            float4* dst = reinterpret_cast<float4*>(g.sk_ws + (size_t)sc.c * kSkSlotFloats + chunk);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(dst + q * 32, make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                               __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
            continue;
          }
          float fa[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) fa[i] = __uint_as_float(v[i]);
          if (finish) {
            for (int d = sc.c + 1; d <= dlast; ++d) {
              const float4* srcp = reinterpret_cast<const float4*>(g.sk_ws + (size_t)d * kSkSlotFloats + chunk);
              float4 p4[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) p4[q] = __ldcg(srcp + q * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                fa[4 * q] += p4[q].x;
                fa[4 * q + 1] += p4[q].y;
                fa[4 * q + 2] += p4[q].z;
                fa[4 * q + 3] += p4[q].w;
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c0 = cb + u * 16;
            const int gc = n0 + c0;
            const int nvalid = min(16, g.Nout - gc);
            if (!rok || nvalid <= 0) continue;
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = fa[16 * u + i];
            if (g.epi == EPI_BF16 && tstore) {
              // 16 values = chunks ch, ch + 1 of the 64-column box bx, 128-byte swizzle
              const int lc = c0 - half * (BN / 2), bx = lc >> 6, ch = (lc & 63) >> 3;
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
              uint8_t* rowp = ostg + bx * 4096 + lane * 128;
              *reinterpret_cast<uint4*>(rowp + ((ch ^ (lane & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              *reinterpret_cast<uint4*>(rowp + (((ch + 1) ^ (lane & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            } else if (g.epi == EPI_BF16) {
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
        }
        if (tstore) {
          // the warp's boxes to global memory; their shared-memory reads finish before the
          // next accumulator is staged over them
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int rowb = m0 + a * (pair ? pair : 128) + wq * 32;
#pragma unroll
            for (int bx = 0; bx < BN / 128; ++bx) {
              const int x = n0 + half * (BN / 2) + bx * 64;
              if (x < g.Nout && rowb < g.M) tma_store_2d(&tmO, x, rowb, smem_u32(ostg) + bx * 4096);
            }
            bulk_commit();
            bulk_wait_read0();
          }
          __syncwarp();
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
      // the B ring held staged output boxes: refill it only once every epilogue warp is done
      if (kOutTma && (s_abort || !mbar_wait(tmemfree, pc & 1))) {
        s_abort = 1;
        break;
      }
      ++pc;
    }
  }

  if (g.out_tma && lane == 0) bulk_wait0();   // this warp's tensor stores have completed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace ls
