// Causal grouped-query attention forward on the 5th-generation tensor core (tcgen05),
// for the decoder layers of the streamed stack (the Llama/Qwen-shaped models the Soup
// pages fine-tune: Soup: Fine-Tune an 8B Model on a 4 GB GPU, "The Core Idea: Layer
// Streaming").
//
// o = softmax(q k^T / sqrt(hd) + causal mask) v per sequence; query head h reads
// key/value head floor(h * kv / nh); the per-row log-sum-exp is saved for the backward.
//
// One CTA owns 128 query rows of one head and walks the key tiles (64 keys each) up to
// the diagonal.  Per key tile j:
//   S_j = Q K_j^T      tcgen05.mma, Q and K_j in shared memory (TMA, 128-byte swizzle),
//                      S_j (128 x 64 fp32) in tensor memory;
//   P_j = exp2(S_j c - m)  the softmax warps read S_j row by row (thread = row) and write
//                      P_j as bf16 into one of two tensor-memory P buffers;
//   O += P_j V_j       tcgen05.mma with A = P_j from tensor memory, B = V_j MN-major in
//                      shared memory, O (128 x hd fp32) in tensor memory.
// S_{j+1} is issued as soon as the softmax warps have read S_j out, so the tensor core
// computes the next scores while they work on this tile; with two P buffers they wait
// for a P V product only to rescale O or to reuse its buffer two tiles later.  K and V
// have rings of their own, each fed by its own producer lane: K_{j+2} needs only S_j to
// be done, V_{j+2} only P_j V_j.  The running maximum m is moved only when a row's
// maximum grows by more than 8 (a factor 256 in the exponentials): O and the row sum l
// are then rescaled together, otherwise both keep the stale m, which changes no result
// since o = O / l and lse = m + log2 l use the same m.
//
// Warps: 0 = TMA producers (lane 0: Q and K, lane 1: V), 1 = tensor-memory owner and MMA
// issuer, 2..5 = softmax and epilogue (warp w reads tensor-memory lanes 32 (w % 4) ..
// + 31).  Every wait is bounded; a timeout raises the device error word and the CTA
// winds down.
#pragma once
#include "attention.cuh"
#include "common.cuh"

namespace ls {

template <int HD>
struct AttnTcCfg {
  static_assert(HD == 64 || HD == 128, "head dim");
  static constexpr int BM = 128;                       // query rows per CTA
  static constexpr int BN = 64;                        // keys per tile
  static constexpr int PANELS = HD / 64;               // 64-column (128 B) panels of a row
  static constexpr int Q_BYTES = BM * HD * 2;          // PANELS x [128 rows x 128 B]
  static constexpr int KV_BYTES = BN * HD * 2;         // one K or V tile: PANELS x [64 rows x 128 B]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;                // K ring: 2 tiles
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;   // V ring: 2 tiles
  static constexpr int OFF_BAR = OFF_V + 2 * KV_BYTES;
  static constexpr int OFF_SLOT = OFF_BAR + 192;
  static constexpr int USED = OFF_BAR + 256 + 1024;    // + slack for the 1 KB alignment
  // at most two CTAs per SM, so that two tensor-memory allocations always fit
  static constexpr int SMEM = USED < 80 * 1024 ? 80 * 1024 : USED;
  static constexpr int TMEM_COLS = 256;
  // column offsets: O, S, two P buffers (bf16 pairs, BN / 2 columns each)
  static constexpr int T_O = 0, T_S = HD, T_P = HD + BN;
  static constexpr int THREADS = 192;
  static_assert(T_P + BN <= TMEM_COLS, "tensor-memory columns");
  // epilogue staging: four warps x 32 padded bf16 rows over the idle Q and K space
  static_assert(4 * 32 * (HD * 2 + 16) <= OFF_V, "output staging");
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int HD>
__global__ void __launch_bounds__(192, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const int* __restrict__ cu, int nh, int nkv,
                       float scale, __nv_bfloat16* __restrict__ out, long long ldo, float* __restrict__ lse, int T,
                       int ntq) {
  using C = AttnTcCfg<HD>;
  extern __shared__ uint8_t attn_tc_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_tc_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(base);
  __shared__ volatile int s_abort;

  const int h = blockIdx.x, s = blockIdx.y;
  const int qt = ntq - 1 - (int)blockIdx.z;   // the longest causal rows start first
  int a, L;
  seq_range(cu, s, T, a, L);
  const int q0 = qt * C::BM;
  if (q0 >= L) return;
  const int g = h / (nh / nkv);
  const int kend = min(L, q0 + C::BM);
  const int nkt = (kend + C::BN - 1) / C::BN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Barriers come in pairs (index b = tile % 2) wherever one side may run a whole tile
  // ahead of the other, so that no waiter can find its phase overtaken by the next one.
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  const uint32_t q_full = bar(0), s_full = bar(9), s_cons = bar(10), drain = bar(15);
  auto k_full = [&](int b) -> uint32_t { return bar(1 + b); };
  auto k_empty = [&](int b) -> uint32_t { return bar(3 + b); };
  auto v_full = [&](int b) -> uint32_t { return bar(5 + b); };
  auto v_empty = [&](int b) -> uint32_t { return bar(7 + b); };
  auto p_full = [&](int b) -> uint32_t { return bar(11 + b); };    // P_j written
  auto pv_done = [&](int b) -> uint32_t { return bar(13 + b); };   // P_j V_j finished

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(k_full(b), 1);
      mbar_init(k_empty(b), 1);
      mbar_init(v_full(b), 1);
      mbar_init(v_empty(b), 1);
      mbar_init(p_full(b), 4);
      mbar_init(pv_done(b), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_cons, 4);
    mbar_init(drain, 1);
    fence_barrier_init();
    s_abort = 0;
    prefetch_tensormap(&tm_qkv);
  }
  if (warp == 1) {
    tmem_alloc(sb + C::OFF_SLOT, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + C::OFF_SLOT);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // lane 0: Q, then the K ring; lane 1: the V ring.  K_j goes into slot j % 2 once S_{j-2}
    // is done, V_j once P_{j-2} V_{j-2} is.
    if (lane < 2) {
      const int xq = h * HD, xk = (nh + g) * HD, xv = (nh + nkv + g) * HD;
      const bool isv = lane == 1;
      if (!isv) {
        mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
        for (int p = 0; p < C::PANELS; ++p)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d(sb + C::OFF_Q + p * 16384 + hf * 8192, &tm_qkv, xq + p * 64, a + q0 + hf * 64, q_full);
      }
      const uint32_t ring = sb + (isv ? C::OFF_V : C::OFF_K);
      const int x = isv ? xv : xk;
      int n = 0;   // tiles issued
      bool ok = true;
      for (int j = 0; j < nkt; ++j) {
        const int b = j & 1;
        if (j >= 2 && (s_abort || !mbar_wait(isv ? v_empty(b) : k_empty(b), ((j - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        const uint32_t fb = isv ? v_full(b) : k_full(b);
        mbar_arrive_expect_tx(fb, C::KV_BYTES);
#pragma unroll
        for (int p = 0; p < C::PANELS; ++p)
          tma_load_2d(ring + b * C::KV_BYTES + p * 8192, &tm_qkv, x + p * 64, a + j * C::BN, fb);
        ++n;
      }
      if (!ok) s_abort = 1;
      // every copy issued has landed before the CTA's shared memory goes away
      if (!isv) mbar_wait(q_full, 0);
      for (int i = n - 2 < 0 ? 0 : n - 2; i < n; ++i) mbar_wait(isv ? v_full(i & 1) : k_full(i & 1), (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16_f32(128, C::BN);
      constexpr uint32_t ID_O = idesc_bf16_f32(128, HD) | (1u << 16);   // B (= V) MN-major
      // S_j = Q K_j^T, then release K slot j % 2
      auto qk = [&](int j) -> bool {
        const int b = j & 1;
        if (s_abort || !mbar_wait(k_full(b), (j >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t kb = sb + C::OFF_K + b * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma_bf16(tmem + C::T_S, sw128_kmajor_desc(sb + C::OFF_Q + (kk >> 2) * 16384 + (kk & 3) * 32),
                      sw128_kmajor_desc(kb + (kk >> 2) * 8192 + (kk & 3) * 32), ID_S, kk > 0 ? 1u : 0u);
        tc_commit(s_full);
        tc_commit(k_empty(b));
        return true;
      };
      bool ok = mbar_wait(q_full, 0) && qk(0);
      for (int j = 0; ok && j < nkt; ++j) {
        const int b = j & 1;
        // S_{j+1} overwrites S_j once the softmax warps have read it out
        if (j + 1 < nkt) ok = !s_abort && mbar_wait(s_cons, j & 1) && qk(j + 1);
        if (!ok || s_abort || !mbar_wait(p_full(b), (j >> 1) & 1) || !mbar_wait(v_full(b), (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vb = sb + C::OFF_V + b * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          tc_mma_bf16_ts(tmem + C::T_O, tmem + C::T_P + b * (C::BN / 2) + kk * 8,
                         sw128_mnmajor_desc(vb + kk * 2048, 8192), ID_O, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(pv_done(b));
        tc_commit(v_empty(b));
      }
      if (!ok) s_abort = 1;
      // every MMA issued has completed before tensor memory is freed
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;                 // tensor-memory lane quarter of this warp
    const int r = q * 32 + lane;            // row of the tile
    const int row = q0 + r;                 // row of the sequence
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    const float c2 = scale * 1.4426950408889634f;   // scores in log2 units
    float m_used = -INFINITY, l = 0.f;
    // a warp-uniform bounded wait: all 32 lanes go on or all stop
    auto wwait = [&](uint32_t b, int par) -> bool {
      const bool good = !s_abort && mbar_wait(b, par);
      return __all_sync(0xffffffffu, good);
    };
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int b = j & 1;
      if (!wwait(s_full, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_32x32b_x32(tl + C::T_S, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld_32x32b_x32(tl + C::T_S + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_cons);
      const int k0 = j * C::BN;
      float x[64];
      float tmax = -INFINITY;
      if (k0 + C::BN - 1 > q0 || k0 + C::BN > L) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int key = k0 + i;
          x[i] = (key > row || key >= L) ? -INFINITY : __uint_as_float(sv[i]);
          tmax = fmaxf(tmax, x[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          x[i] = __uint_as_float(sv[i]);
          tmax = fmaxf(tmax, x[i]);
        }
      }
      const float m_new = fmaxf(m_used, tmax * c2);
      const bool resc = m_new > m_used + 8.f;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      float sum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2_approx(fmaf(x[2 * i], c2, -m_used));
        const float p1 = ex2_approx(fmaf(x[2 * i + 1], c2, -m_used));
        sum += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + sum;
      // P buffer j % 2 was last read by P_{j-2} V_{j-2}
      if (j >= 2) {
        if (!wwait(pv_done(b), ((j - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // O is rescaled once it holds P_{j-1} V_{j-1}
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        if (!wwait(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tl + C::T_O + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_32x32b_x32(tl + C::T_O + c * 32, o);
        }
      }
      tmem_st_32x32b_x32(tl + C::T_P + b * (C::BN / 2), pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(b));
    }
    if (ok) ok = wwait(pv_done((nkt - 1) & 1), ((nkt - 1) >> 1) & 1);
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      // O / l as bf16 rows, staged in this warp's part of the (now idle) Q / K space, then
      // written out a row at a time by the whole warp (coalesced)
      constexpr int RS = HD * 2 + 16;   // padded row: consecutive lanes hit different banks
      uint8_t* stg = base + C::OFF_Q + q * 32 * RS;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tl + C::T_O + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
          *reinterpret_cast<uint4*>(stg + lane * RS + c * 64 + v * 16) = w;
        }
      }
      if (row < L) lse[(size_t)h * T + a + row] = (m_used + log2f(l)) * 0.6931471805599453f;
      __syncwarp();
      const int rlast = min(32, L - (q0 + q * 32));   // rows of this warp inside the sequence
      for (int i = 0; i < rlast; ++i) {
        __nv_bfloat16* orow = out + (size_t)(a + q0 + q * 32 + i) * ldo + (size_t)h * HD;
        if constexpr (HD == 128)
          *reinterpret_cast<uint2*>(orow + lane * 4) = *reinterpret_cast<const uint2*>(stg + i * RS + lane * 8);
        else
          *reinterpret_cast<uint32_t*>(orow + lane * 2) = *reinterpret_cast<const uint32_t*>(stg + i * RS + lane * 4);
      }
    } else {
      s_abort = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ backward
// With P = exp(S / sqrt(hd) - lse) (the forward's saved log-sum-exp) and
// D = rowsum(dO o O):  dS = P o (dP - D), dP = dO V^T;
//   dQ = dS K / sqrt(hd),  dK = dS^T Q / sqrt(hd),  dV = P^T dO.
// Two kernels, each deterministic (every output element is summed by one CTA in a fixed
// order): dQ per 128-query tile and head over the key tiles up to the diagonal; dK, dV
// per 128-key tile over the query tiles from the diagonal on and the query heads of one
// slice of the key/value group.  S and dP are recomputed in each.

template <int HD>
struct AttnBwdTcCfg {
  static_assert(HD == 64 || HD == 128, "head dim");
  static constexpr int PANELS = HD / 64;
  static constexpr int T128 = 128 * HD * 2;   // 128 rows x HD (PANELS x [128 rows x 128 B])
  static constexpr int T64 = 64 * HD * 2;     // 64 rows x HD  (PANELS x [64 rows x 128 B])
  // dQ kernel: Q, dO (128 query rows); stages of (K, V) (64 keys)
  static constexpr int NST = 3;               // stages of the streamed operand ring
  static constexpr int Q_OFF_Q = 0, Q_OFF_DO = T128, Q_OFF_KV = 2 * T128;
  static constexpr int Q_OFF_BAR = Q_OFF_KV + NST * 2 * T64;
  // dK/dV kernel: K, V (128 keys); stages of (Q, dO) (64 query rows), then lse / D rows
  static constexpr int K_OFF_K = 0, K_OFF_V = T128, K_OFF_QD = 2 * T128;
  static constexpr int K_OFF_BAR = K_OFF_QD + NST * 2 * T64;
  static constexpr int OFF_SLOT = 192;                 // tensor-memory address, after the barriers
  static constexpr int BAR_BYTES = 256;
  // one CTA per SM: each takes all 512 tensor-memory columns
  static constexpr int SMEM_Q = (Q_OFF_BAR + BAR_BYTES + 1024) < 116 * 1024 ? 116 * 1024 : Q_OFF_BAR + BAR_BYTES + 1024;
  static constexpr int SMEM_K = (K_OFF_BAR + BAR_BYTES + 1024) < 116 * 1024 ? 116 * 1024 : K_OFF_BAR + BAR_BYTES + 1024;
  static constexpr int TMEM_COLS = 512;
  // dQ kernel columns: dQ, S x2, dP x2, dS x2 (bf16 pairs)
  static constexpr int DQ_ACC = 0, DQ_S = HD, DQ_DP = HD + 128, DQ_DS = HD + 256;
  // dK/dV kernel columns: dK, dV, S^T, dP^T, P^T x2, dS^T x2
  static constexpr int KV_DK = 0, KV_DV = HD, KV_S = 2 * HD, KV_DP = 2 * HD + 64, KV_P = 2 * HD + 128,
                       KV_DS = 2 * HD + 192;
  // warps 2..9: two per tensor-memory lane quarter, each taking one half (32) of a tile's
  // 64 columns, so that every SM sub-partition runs two of them
  static constexpr int THREADS = 64 + 256;
  static constexpr int NSOFT = 8;
  // epilogue staging: eight warps x 32 padded rows over the idle operand space
  static_assert(8 * 32 * (HD * 2 + 16) <= Q_OFF_BAR && 8 * 32 * (128 + 16) <= K_OFF_BAR, "output staging");
};

template <int HD>
__global__ void __launch_bounds__(AttnBwdTcCfg<HD>::THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                          const float* __restrict__ lse, const float* __restrict__ Dd, const int* __restrict__ cu,
                          int nh, int nkv, float scale, float* __restrict__ dqkv, long long ldg, int T, int ntq) {
  using C = AttnBwdTcCfg<HD>;
  extern __shared__ uint8_t attn_tc_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_tc_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(base);
  __shared__ volatile int s_abort;

  const int h = blockIdx.x, s = blockIdx.y;
  const int qt = ntq - 1 - (int)blockIdx.z;
  int a, L;
  seq_range(cu, s, T, a, L);
  const int q0 = qt * 128;
  if (q0 >= L) return;
  const int g = h / (nh / nkv);
  const int kend = min(L, q0 + 128);
  const int nkt = (kend + 63) / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bars = sb + C::Q_OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8 * i; };
  constexpr int NST = C::NST;
  const uint32_t q_full = bar(0), drain = bar(15);
  auto kv_full = [&](int st) -> uint32_t { return bar(1 + st); };    // K_j, V_j in stage j % NST
  auto kv_empty = [&](int st) -> uint32_t { return bar(4 + st); };
  auto sd_full = [&](int b) -> uint32_t { return bar(7 + b); };    // S_j, dP_j computed, j % 2 = b
  auto sd_free = [&](int b) -> uint32_t { return bar(9 + b); };    // ... and read out
  auto ds_full = [&](int b) -> uint32_t { return bar(11 + b); };   // dS_j written
  auto ds_done = [&](int b) -> uint32_t { return bar(13 + b); };   // dQ += dS_j K_j finished

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int st = 0; st < NST; ++st) {
      mbar_init(kv_full(st), 1);
      mbar_init(kv_empty(st), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sd_full(b), 1);
      mbar_init(sd_free(b), C::NSOFT);
      mbar_init(ds_full(b), C::NSOFT);
      mbar_init(ds_done(b), 1);
    }
    mbar_init(drain, 1);
    fence_barrier_init();
    s_abort = 0;
    prefetch_tensormap(&tm_qkv);
    prefetch_tensormap(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(bars + C::OFF_SLOT, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + C::Q_OFF_BAR + C::OFF_SLOT);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int xq = h * HD, xk = (nh + g) * HD, xv = (nh + nkv + g) * HD;
      mbar_arrive_expect_tx(q_full, 2 * C::T128);
#pragma unroll
      for (int p = 0; p < C::PANELS; ++p)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tma_load_2d(sb + C::Q_OFF_Q + p * 16384 + hf * 8192, &tm_qkv, xq + p * 64, a + q0 + hf * 64, q_full);
          tma_load_2d(sb + C::Q_OFF_DO + p * 16384 + hf * 8192, &tm_do, xq + p * 64, a + q0 + hf * 64, q_full);
        }
      int j = 0;
      bool ok = true;
      for (; j < nkt; ++j) {
        const int st = j % NST;
        if (j >= NST && (s_abort || !mbar_wait(kv_empty(st), ((j / NST) - 1) & 1))) {
          ok = false;
          break;
        }
        const uint32_t kb = sb + C::Q_OFF_KV + st * 2 * C::T64, vb = kb + C::T64;
        mbar_arrive_expect_tx(kv_full(st), 2 * C::T64);
#pragma unroll
        for (int p = 0; p < C::PANELS; ++p) {
          tma_load_2d(kb + p * 8192, &tm_qkv, xk + p * 64, a + j * 64, kv_full(st));
          tma_load_2d(vb + p * 8192, &tm_qkv, xv + p * 64, a + j * 64, kv_full(st));
        }
      }
      if (!ok) s_abort = 1;
      mbar_wait(q_full, 0);
      for (int i = j - NST < 0 ? 0 : j - NST; i < j; ++i) mbar_wait(kv_full(i % NST), (i / NST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16_f32(128, 64);
      constexpr uint32_t ID_Q = idesc_bf16_f32(128, HD) | (1u << 16);   // B (= K) MN-major
      // dQ += dS_i K_i, then release dS buffer i % 2 and stage i's K/V
      auto dq = [&](int i) -> bool {
        if (s_abort || !mbar_wait(ds_full(i & 1), (i >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t kb = sb + C::Q_OFF_KV + (i % NST) * 2 * C::T64;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16_ts(tmem + C::DQ_ACC, tmem + C::DQ_DS + (i & 1) * 32 + kk * 8,
                         sw128_mnmajor_desc(kb + kk * 2048, 8192), ID_Q, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(ds_done(i & 1));
        tc_commit(kv_empty(i % NST));
        return true;
      };
      bool ok = mbar_wait(q_full, 0);
      for (int j = 0; ok && j < nkt; ++j) {
        const int b = j & 1;
        if (s_abort || !mbar_wait(kv_full(j % NST), (j / NST) & 1) ||
            (j >= 2 && !mbar_wait(sd_free(b), ((j - 2) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = sb + C::Q_OFF_KV + (j % NST) * 2 * C::T64, vb = kb + C::T64;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32, koff = (kk >> 2) * 8192 + (kk & 3) * 32;
          tc_mma_bf16(tmem + C::DQ_S + b * 64, sw128_kmajor_desc(sb + C::Q_OFF_Q + off), sw128_kmajor_desc(kb + koff),
                      ID_S, kk > 0 ? 1u : 0u);
          tc_mma_bf16(tmem + C::DQ_DP + b * 64, sw128_kmajor_desc(sb + C::Q_OFF_DO + off),
                      sw128_kmajor_desc(vb + koff), ID_S, kk > 0 ? 1u : 0u);
        }
        tc_commit(sd_full(b));
        if (j > 0) ok = dq(j - 1);
      }
      if (ok) ok = dq(nkt - 1);
      if (!ok) s_abort = 1;
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ dS + epilogue
    const int qw = warp & 3, hf = (warp - 2) >> 2;   // lane quarter, column half
    const int row = q0 + qw * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    const float c2 = scale * 1.4426950408889634f;
    // rows past the sequence get P = 0 (exp2(-inf))
    const float lse2 = row < L ? lse[(size_t)h * T + a + row] * 1.4426950408889634f : INFINITY;
    const float drow = row < L ? Dd[(size_t)h * T + a + row] : 0.f;
    auto wwait = [&](uint32_t b, int par) -> bool {
      const bool good = !s_abort && mbar_wait(b, par);
      return __all_sync(0xffffffffu, good);
    };
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int b = j & 1;
      if (!wwait(sd_full(b), (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[32], dp[32];
      tmem_ld_32x32b_x32(tl + C::DQ_S + b * 64 + hf * 32, sv);
      tmem_ld_32x32b_x32(tl + C::DQ_DP + b * 64 + hf * 32, dp);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sd_free(b));
      const int k0 = j * 64 + hf * 32;   // first key of this thread's half
      const bool edge = k0 + 31 > q0 || k0 + 32 > L;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float d2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = 2 * i + e;
          float pr = ex2_approx(fmaf(__uint_as_float(sv[c]), c2, -lse2));
          if (edge && (k0 + c > row || k0 + c >= L)) pr = 0.f;
          d2[e] = pr * (__uint_as_float(dp[c]) - drow);
        }
        pk[i] = pack_bf16x2(d2[0], d2[1]);
      }
      // dS buffer j % 2 was last read by dQ += dS_{j-2} K_{j-2}
      if (j >= 2) {
        if (!wwait(ds_done(b), ((j - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st_32x32b_x16(tl + C::DQ_DS + b * 32 + hf * 16, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full(b));
    }
    if (ok) ok = wwait(ds_done((nkt - 1) & 1), ((nkt - 1) >> 1) & 1);
    if (ok) {
      tc_fence_after();
      // this warp's half of its 32 dQ rows, staged in the idle Q / dO / K / V space, then
      // written out a row at a time by the whole warp (coalesced)
      constexpr int HB = HD * 2;        // bytes of a half row (HD / 2 fp32)
      constexpr int RS = HB + 16;
      uint8_t* stg = base + (warp - 2) * 32 * RS;
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tl + C::DQ_ACC + hf * (HD / 2) + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *reinterpret_cast<float4*>(stg + lane * RS + c * 128 + v * 16) =
              make_float4(__uint_as_float(o[4 * v]) * scale, __uint_as_float(o[4 * v + 1]) * scale,
                          __uint_as_float(o[4 * v + 2]) * scale, __uint_as_float(o[4 * v + 3]) * scale);
      }
      __syncwarp();
      const int rlast = min(32, L - (q0 + qw * 32));
      for (int i = 0; i < rlast; ++i) {
        float* grow = dqkv + (size_t)(a + q0 + qw * 32 + i) * ldg + (size_t)h * HD + hf * (HD / 2);
        if constexpr (HD == 128)
          *reinterpret_cast<float2*>(grow + lane * 2) = *reinterpret_cast<const float2*>(stg + i * RS + lane * 8);
        else
          grow[lane] = *reinterpret_cast<const float*>(stg + i * RS + lane * 4);
      }
    } else {
      s_abort = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// grid (nkv * hsplit, nseq, ceil(maxlen / 128)), the key tiles with the most query tiles
// first.  hsplit > 1: this CTA takes one slice of the group's query heads and writes its
// dK (scaled) and dV to part [hsplit][T][2 nkv HD] for attn_dkdv_reduce_kernel; otherwise
// into dqkv.  The producer warp also stages each query tile's lse and D rows in shared
// memory (each lane two of each, then an arrive on the tile's barrier).
template <int HD>
__global__ void __launch_bounds__(AttnBwdTcCfg<HD>::THREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                            const float* __restrict__ lse, const float* __restrict__ Dd, const int* __restrict__ cu,
                            int nh, int nkv, float scale, float* __restrict__ dqkv, long long ldg, int T, int hsplit,
                            float* __restrict__ part) {
  using C = AttnBwdTcCfg<HD>;
  extern __shared__ uint8_t attn_tc_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_tc_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(base);
  __shared__ volatile int s_abort;
  __shared__ __align__(16) float s_ld[C::NST][2][64];   // per query-tile stage: lse (log2 units), D

  const int s = blockIdx.y, g = blockIdx.x / hsplit, hs = blockIdx.x % hsplit;
  int a, L;
  seq_range(cu, s, T, a, L);
  const int k0 = blockIdx.z * 128;
  if (k0 >= L) return;
  const int group = nh / nkv;
  const int per = (group + hsplit - 1) / hsplit;
  const int h_lo = g * group + hs * per;
  const int nheads = max(0, min(per, group - hs * per));
  const int nqt = (L - k0 + 63) / 64;          // query tiles from the diagonal on
  const int nit = nheads * nqt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bars = sb + C::K_OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8 * i; };
  constexpr int NST = C::NST;
  const uint32_t kv_full = bar(0), st_full = bar(7), st_free = bar(8), drain = bar(13);
  auto qd_full = [&](int st) -> uint32_t { return bar(1 + st); };   // Q_i, dO_i (+ lse, D) in stage i % NST
  auto qd_empty = [&](int st) -> uint32_t { return bar(4 + st); };
  auto pd_full = [&](int b) -> uint32_t { return bar(9 + b); };    // P^T_i, dS^T_i written, i % 2 = b
  auto pd_done = [&](int b) -> uint32_t { return bar(11 + b); };   // dV, dK products of tile i finished

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int st = 0; st < NST; ++st) {
      mbar_init(qd_full(st), 1 + 32);   // the TMA bytes, and the producer lanes' lse / D stores
      mbar_init(qd_empty(st), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(pd_full(b), C::NSOFT);
      mbar_init(pd_done(b), 1);
    }
    mbar_init(st_full, 1);
    mbar_init(st_free, C::NSOFT);
    mbar_init(drain, 1);
    fence_barrier_init();
    s_abort = 0;
    prefetch_tensormap(&tm_qkv);
    prefetch_tensormap(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(bars + C::OFF_SLOT, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + C::K_OFF_BAR + C::OFF_SLOT);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (whole warp)
    if (nit > 0) {
      const int xk = (nh + g) * HD, xv = (nh + nkv + g) * HD;
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::T128);
#pragma unroll
        for (int p = 0; p < C::PANELS; ++p)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_2d(sb + C::K_OFF_K + p * 16384 + hf * 8192, &tm_qkv, xk + p * 64, a + k0 + hf * 64, kv_full);
            tma_load_2d(sb + C::K_OFF_V + p * 16384 + hf * 8192, &tm_qkv, xv + p * 64, a + k0 + hf * 64, kv_full);
          }
      }
      int i = 0;
      bool ok = true;
      for (; i < nit; ++i) {
        const int b = i % NST;
        bool good = true;
        if (i >= NST) good = !s_abort && mbar_wait(qd_empty(b), ((i / NST) - 1) & 1);
        if (!__all_sync(0xffffffffu, good)) {
          ok = false;
          break;
        }
        const int h = h_lo + i / nqt, q0 = k0 + (i % nqt) * 64;
        if (lane == 0) {
          const uint32_t qb = sb + C::K_OFF_QD + b * 2 * C::T64, ob = qb + C::T64;
          mbar_arrive_expect_tx(qd_full(b), 2 * C::T64);
#pragma unroll
          for (int p = 0; p < C::PANELS; ++p) {
            tma_load_2d(qb + p * 8192, &tm_qkv, h * HD + p * 64, a + q0, qd_full(b));
            tma_load_2d(ob + p * 8192, &tm_do, h * HD + p * 64, a + q0, qd_full(b));
          }
        }
        // lse in log2 units (+inf past the sequence, so that P = 0 there) and D
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = lane + 32 * e, q = q0 + c;
          s_ld[b][0][c] = q < L ? lse[(size_t)h * T + a + q] * 1.4426950408889634f : INFINITY;
          s_ld[b][1][c] = q < L ? Dd[(size_t)h * T + a + q] : 0.f;
        }
        mbar_arrive(qd_full(b));
      }
      if (lane == 0) {
        if (!ok) s_abort = 1;
        mbar_wait(kv_full, 0);
        for (int j = i - NST < 0 ? 0 : i - NST; j < i; ++j) mbar_wait(qd_full(j % NST), (j / NST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nit > 0) {
      constexpr uint32_t ID_S = idesc_bf16_f32(128, 64);
      constexpr uint32_t ID_O = idesc_bf16_f32(128, HD) | (1u << 16);   // B (= dO, Q) MN-major
      // dV += P^T_i dO_i, dK += dS^T_i Q_i, then release buffers i % 2
      auto kv = [&](int i) -> bool {
        if (s_abort || !mbar_wait(pd_full(i & 1), (i >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t qb = sb + C::K_OFF_QD + (i % NST) * 2 * C::T64, ob = qb + C::T64;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc_mma_bf16_ts(tmem + C::KV_DV, tmem + C::KV_P + (i & 1) * 32 + kk * 8,
                         sw128_mnmajor_desc(ob + kk * 2048, 8192), ID_O, (i > 0 || kk > 0) ? 1u : 0u);
          tc_mma_bf16_ts(tmem + C::KV_DK, tmem + C::KV_DS + (i & 1) * 32 + kk * 8,
                         sw128_mnmajor_desc(qb + kk * 2048, 8192), ID_O, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(pd_done(i & 1));
        tc_commit(qd_empty(i % NST));
        return true;
      };
      bool ok = mbar_wait(kv_full, 0);
      for (int i = 0; ok && i < nit; ++i) {
        // S^T, dP^T of tile i overwrite tile i-1's: the softmax warps must have read them
        if (s_abort || !mbar_wait(qd_full(i % NST), (i / NST) & 1) || (i > 0 && !mbar_wait(st_free, (i - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t qb = sb + C::K_OFF_QD + (i % NST) * 2 * C::T64, ob = qb + C::T64;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32, qoff = (kk >> 2) * 8192 + (kk & 3) * 32;
          tc_mma_bf16(tmem + C::KV_S, sw128_kmajor_desc(sb + C::K_OFF_K + off), sw128_kmajor_desc(qb + qoff), ID_S,
                      kk > 0 ? 1u : 0u);
          tc_mma_bf16(tmem + C::KV_DP, sw128_kmajor_desc(sb + C::K_OFF_V + off), sw128_kmajor_desc(ob + qoff), ID_S,
                      kk > 0 ? 1u : 0u);
        }
        tc_commit(st_full);
        if (i > 0) ok = kv(i - 1);
      }
      if (ok) ok = kv(nit - 1);
      if (!ok) s_abort = 1;
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ P^T, dS^T + epilogue
    const int qw = warp & 3, hf = (warp - 2) >> 2;   // lane quarter, column half
    const int key = k0 + qw * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(qw * 32) << 16);
    const float c2 = scale * 1.4426950408889634f;
    auto wwait = [&](uint32_t b, int par) -> bool {
      const bool good = !s_abort && mbar_wait(b, par);
      return __all_sync(0xffffffffu, good);
    };
    bool ok = true;
    for (int i = 0; i < nit; ++i) {
      const int b = i & 1;
      // the tile's lse / D rows are in shared memory once its stage is full
      if (!wwait(qd_full(i % NST), (i / NST) & 1) || !wwait(st_full, i & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[32], dp[32];
      tmem_ld_32x32b_x32(tl + C::KV_S + hf * 32, sv);
      tmem_ld_32x32b_x32(tl + C::KV_DP + hf * 32, dp);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(st_free);
      const int q0 = k0 + (i % nqt) * 64 + hf * 32;   // first query of this thread's half
      const bool diag = q0 < k0 + 128;                // the half crosses the diagonal
      const float* sl = s_ld[i % NST][0] + hf * 32;
      const float* sd = s_ld[i % NST][1] + hf * 32;
      uint32_t pp[16], pd[16];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l4 = *reinterpret_cast<const float4*>(sl + 4 * c4);
        const float4 d4 = *reinterpret_cast<const float4*>(sd + 4 * c4);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
        float pr[4], ds[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 4 * c4 + e;
          float x = ex2_approx(fmaf(__uint_as_float(sv[c]), c2, -lv[e]));
          if (diag && q0 + c < key) x = 0.f;
          pr[e] = x;
          ds[e] = x * (__uint_as_float(dp[c]) - dv[e]);
        }
        pp[2 * c4] = pack_bf16x2(pr[0], pr[1]);
        pp[2 * c4 + 1] = pack_bf16x2(pr[2], pr[3]);
        pd[2 * c4] = pack_bf16x2(ds[0], ds[1]);
        pd[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
      }
      // buffers i % 2 were last read by the products of tile i-2
      if (i >= 2) {
        if (!wwait(pd_done(b), ((i - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st_32x32b_x16(tl + C::KV_P + b * 32 + hf * 16, pp);
      tmem_st_32x32b_x16(tl + C::KV_DS + b * 32 + hf * 16, pd);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pd_full(b));
    }
    if (ok && nit > 0) ok = wwait(pd_done((nit - 1) & 1), ((nit - 1) >> 1) & 1);
    if (ok) {
      if (nit > 0) tc_fence_after();
      // half 0 writes dK, half 1 dV: HD / 64 passes of 32 columns per row, each staged in
      // this warp's part of the idle K / V / Q / dO space and written out a row at a time
      // by the whole warp (coalesced)
      {
        const int w = hf;
        const float f = w == 0 ? scale : 1.f;
        constexpr int RS = 128 + 16;
        uint8_t* stg = base + (warp - 2) * 32 * RS;
        const int rlast = min(32, L - (k0 + qw * 32));
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          if (nit > 0) {
            tmem_ld_32x32b_x32(tl + (w == 0 ? C::KV_DK : C::KV_DV) + c * 32, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int v = 0; v < 32; ++v) o[v] = 0u;
          }
          __syncwarp();   // the previous pass's rows have been read out
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(stg + lane * RS + v * 16) =
                make_float4(__uint_as_float(o[4 * v]) * f, __uint_as_float(o[4 * v + 1]) * f,
                            __uint_as_float(o[4 * v + 2]) * f, __uint_as_float(o[4 * v + 3]) * f);
          __syncwarp();
          for (int i = 0; i < rlast; ++i) {
            const int kr = k0 + qw * 32 + i;
            float* dst = hsplit > 1
                             ? part + ((size_t)hs * T + a + kr) * (2 * nkv * HD) + (size_t)(w * nkv + g) * HD
                             : dqkv + (size_t)(a + kr) * ldg + (size_t)(nh + w * nkv + g) * HD;
            dst[c * 32 + lane] = *reinterpret_cast<const float*>(stg + i * RS + lane * 4);
          }
        }
      }
    } else {
      s_abort = 1;
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
