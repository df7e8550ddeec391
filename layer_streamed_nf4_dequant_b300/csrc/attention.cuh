// Causal grouped-query attention, forward and backward, for the decoder layers of
// the streamed stack (the Llama/Qwen-shaped models the Soup pages fine-tune:
// Soup: Fine-Tune an 8B Model on a 4 GB GPU, "The Core Idea: Layer Streaming").
//
// o = softmax(q k^T / sqrt(hd) + causal mask) v per sequence; query head h reads
// key/value head floor(h * kv / nh).  Online softmax over 64-key tiles (the score
// matrix is never stored); the forward saves the per-row log-sum-exp.  The backward
// is deterministic: one kernel accumulates dq per query tile, another dk/dv per key
// tile summing over the query heads of its group in a fixed order (no atomics).
// Matrix products use bf16 tensor-core MMA (m16n8k16) with fp32 accumulation.
#pragma once
#include "common.cuh"

namespace ls {

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// A fragment (16 x 16) from a row-major smem tile: rows m0.., cols k0..
__device__ __forceinline__ void ldsm_A(uint32_t (&r)[4], const __nv_bfloat16* base, int ld, int m0, int k0,
                                       int lane) {
  ldsm_x4(r, base + (m0 + (lane & 15)) * ld + k0 + ((lane >> 4) << 3));
}
// B fragments for n-tiles n0/8 and n0/8+1 at k-step k0, smem rows indexed by n, cols by k.
__device__ __forceinline__ void ldsm_B_nk(uint32_t (&r)[4], const __nv_bfloat16* base, int ld, int n0, int k0,
                                          int lane) {
  const int i = lane >> 3;
  ldsm_x4(r, base + (n0 + ((i >> 1) << 3) + (lane & 7)) * ld + k0 + ((i & 1) << 3));
}
// Same, smem rows indexed by k, cols by n (transposing load).
__device__ __forceinline__ void ldsm_B_kn(uint32_t (&r)[4], const __nv_bfloat16* base, int ld, int k0, int n0,
                                          int lane) {
  const int i = lane >> 3;
  ldsm_x4_t(r, base + (k0 + ((i & 1) << 3) + (lane & 7)) * ld + n0 + ((i >> 1) << 3));
}
// Accumulator tiles 2kk, 2kk+1 (16 x 8 each) as one bf16 A fragment over 16 columns.
__device__ __forceinline__ void acc_to_A(uint32_t (&a)[4], const float (&c0)[4], const float (&c1)[4]) {
  a[0] = pack_bf16x2(c0[0], c0[1]);
  a[1] = pack_bf16x2(c0[2], c0[3]);
  a[2] = pack_bf16x2(c1[0], c1[1]);
  a[3] = pack_bf16x2(c1[2], c1[3]);
}

template <int HD>
__device__ __forceinline__ void load_tile(__nv_bfloat16* dst, const __nv_bfloat16* src, long long ld, int r0,
                                          int L, int tid, int nthr) {
  constexpr int LDS = HD + 8;
  for (int e = tid; e < 64 * (HD / 8); e += nthr) {
    const int r = e / (HD / 8), c = e % (HD / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r0 + r < L) v = *reinterpret_cast<const uint4*>(src + (size_t)(r0 + r) * ld + c * 8);
    *reinterpret_cast<uint4*>(dst + r * LDS + c * 8) = v;
  }
}

// Asynchronous variant: 16-byte cp.async per chunk, rows at or past L zero-filled (source
// size 0, no global read).  The caller commits the group and waits on it.
template <int HD>
__device__ __forceinline__ void load_tile_async(__nv_bfloat16* dst, const __nv_bfloat16* src, long long ld, int r0,
                                                int L, int tid, int nthr) {
  constexpr int LDS = HD + 8;
  for (int e = tid; e < 64 * (HD / 8); e += nthr) {
    const int r = e / (HD / 8), c = e % (HD / 8);
    const bool ok = r0 + r < L;
    const __nv_bfloat16* g = ok ? src + (size_t)(r0 + r) * ld + c * 8 : src;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + r * LDS + c * 8)), "l"(g),
                 "r"(ok ? 16 : 0)
                 : "memory");
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ forward
// grid (ceil(maxlen / 64), nh, nseq), 128 threads: warp w owns query rows 16w..16w+15.
// Rows [a, a + L) of sequence s.  The offsets come from the caller; a list that is not
// 0 <= cu[s] <= cu[s+1] <= T is clamped into the batch and raises the device error word,
// so a malformed batch cannot make a kernel read or write outside its buffers.
__device__ __forceinline__ void seq_range(const int* __restrict__ cu, int s, int T, int& a, int& L) {
  int x = cu[s], y = cu[s + 1];
  if (x < 0 || y < x || y > T) {
    raise_error(DEV_BAD_ARG);
    x = min(max(x, 0), T);
    y = min(max(y, x), T);
  }
  a = x;
  L = y - x;
}

template <int HD>
__global__ void __launch_bounds__(128) attn_fwd_kernel(const __nv_bfloat16* __restrict__ qkv, long long ld,
                                                       const int* __restrict__ cu, int nh, int nkv, float scale,
                                                       __nv_bfloat16* __restrict__ out, long long ldo,
                                                       float* __restrict__ lse, int T) {
  constexpr int LDS = HD + 8;
  extern __shared__ __align__(16) uint8_t attn_smem[];
  // Q, then two (K, V) buffers: the next key tile is copied while this one computes
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(attn_smem);
  const int s = blockIdx.z, h = blockIdx.y;
  int a, L;
  seq_range(cu, s, T, a, L);
  const int q0 = blockIdx.x * 64;
  if (q0 >= L) return;
  const int g = h / (nh / nkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const __nv_bfloat16* Qg = qkv + (size_t)a * ld + (size_t)h * HD;
  const __nv_bfloat16* Kg = qkv + (size_t)a * ld + (size_t)(nh + g) * HD;
  const __nv_bfloat16* Vg = qkv + (size_t)a * ld + (size_t)(nh + nkv + g) * HD;
  load_tile_async<HD>(sQ, Qg, ld, q0, L, tid, 128);
  load_tile_async<HD>(sQ + 64 * LDS, Kg, ld, 0, L, tid, 128);
  load_tile_async<HD>(sQ + 2 * 64 * LDS, Vg, ld, 0, L, tid, 128);
  cp_async_commit();
  const float c2 = scale * kLog2e;
  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int row0 = q0 + warp * 16 + (lane >> 2);
  const int kend = min(L, q0 + 64);
  for (int k0 = 0, it = 0; k0 < kend; k0 += 64, ++it) {
    __nv_bfloat16* sK = sQ + (1 + 2 * (it & 1)) * 64 * LDS;
    __nv_bfloat16* sV = sK + 64 * LDS;
    if (k0 + 64 < kend) {
      __nv_bfloat16* nK = sQ + (1 + 2 * ((it + 1) & 1)) * 64 * LDS;
      load_tile_async<HD>(nK, Kg, ld, k0 + 64, L, tid, 128);
      load_tile_async<HD>(nK + 64 * LDS, Vg, ld, k0 + 64, L, tid, 128);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    float sc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD; ks += 16) {
      uint32_t af[4];
      ldsm_A(af, sQ, LDS, warp * 16, ks, lane);
#pragma unroll
      for (int nt = 0; nt < 8; nt += 2) {
        uint32_t b[4];
        ldsm_B_nk(b, sK, LDS, nt * 8, ks, lane);
        mma16816(sc[nt], af, b[0], b[1]);
        mma16816(sc[nt + 1], af, b[2], b[3]);
      }
    }
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k0 + nt * 8 + 2 * (lane & 3) + (e & 1);
        const int row = row0 + (e >> 1) * 8;
        float v = sc[nt][e] * c2;
        if (key > row || key >= L) v = -INFINITY;
        sc[nt][e] = v;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
      }
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
      const float mn = fmaxf(mrow[r], tmax[r]);
      alpha[r] = (mn == -INFINITY) ? 1.f : exp2f(mrow[r] - mn);
      mrow[r] = mn;
      lrow[r] *= alpha[r];
    }
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
      o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float m = mrow[e >> 1];
        const float p = (sc[nt][e] == -INFINITY) ? 0.f : exp2f(sc[nt][e] - m);
        sc[nt][e] = p;
        lrow[e >> 1] += p;
      }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      acc_to_A(pa, sc[2 * kk], sc[2 * kk + 1]);
#pragma unroll
      for (int dn = 0; dn < HD / 8; dn += 2) {
        uint32_t b[4];
        ldsm_B_kn(b, sV, LDS, kk * 16, dn * 8, lane);
        mma16816(o[dn], pa, b[0], b[1]);
        mma16816(o[dn + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();   // every warp is done with this buffer before it is refilled
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = row0 + r * 8;
    if (row >= L) continue;
    const float inv = 1.f / lrow[r];
    __nv_bfloat16* orow = out + (size_t)(a + row) * ldo + (size_t)h * HD;
#pragma unroll
    for (int dn = 0; dn < HD / 8; ++dn) {
      const int col = dn * 8 + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(orow + col) = pack_bf16x2(o[dn][2 * r] * inv, o[dn][2 * r + 1] * inv);
    }
    if ((lane & 3) == 0) lse[(size_t)h * T + a + row] = (mrow[r] + log2f(lrow[r])) * kLn2;
  }
}

// D[h, t] = sum_d dO[t, h, d] * O[t, h, d]   (one warp per (t, h))
__global__ void attn_bwd_dot_kernel(const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ o,
                                    long long ld, int nh, int hd, float* __restrict__ D, int T) {
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= T * nh) return;
  const int t = w / nh, h = w % nh;
  const __nv_bfloat16* a = dout + (size_t)t * ld + (size_t)h * hd;
  const __nv_bfloat16* b = o + (size_t)t * ld + (size_t)h * hd;
  float acc = 0.f;
  // four consecutive elements per lane (8-byte reads; hd and ld are multiples of 4)
  for (int d = lane * 4; d < hd; d += 128) {
    const uint2 x = *reinterpret_cast<const uint2*>(a + d), y = *reinterpret_cast<const uint2*>(b + d);
    acc += bf16lo(x.x) * bf16lo(y.x);
    acc += bf16hi(x.x) * bf16hi(y.x);
    acc += bf16lo(x.y) * bf16lo(y.y);
    acc += bf16hi(x.y) * bf16hi(y.y);
  }
  acc = warp_sum(acc);
  if (lane == 0) D[(size_t)h * T + t] = acc;
}

// ------------------------------------------------------------------ backward: dq
// grid (ceil(maxlen / 64), nh, nseq).  dq written (fp32) into dqkv_f's q columns.
template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const __nv_bfloat16* __restrict__ qkv, long long ld,
                                                          const __nv_bfloat16* __restrict__ dout, long long lddo,
                                                          const float* __restrict__ lse, const float* __restrict__ D,
                                                          const int* __restrict__ cu, int nh, int nkv, float scale,
                                                          float* __restrict__ dqkv, long long ldg, int T) {
  constexpr int LDS = HD + 8;
  extern __shared__ __align__(16) uint8_t attn_smem[];
  // Q, dO, then two (K, V) buffers (the next key tile is copied while this one computes)
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(attn_smem);
  __nv_bfloat16* sO = sQ + 64 * LDS;
  const int s = blockIdx.z, h = blockIdx.y;
  int a, L;
  seq_range(cu, s, T, a, L);
  const int q0 = blockIdx.x * 64;
  if (q0 >= L) return;
  const int g = h / (nh / nkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const __nv_bfloat16* Kg = qkv + (size_t)a * ld + (size_t)(nh + g) * HD;
  const __nv_bfloat16* Vg = qkv + (size_t)a * ld + (size_t)(nh + nkv + g) * HD;
  load_tile_async<HD>(sQ, qkv + (size_t)a * ld + (size_t)h * HD, ld, q0, L, tid, 128);
  load_tile_async<HD>(sO, dout + (size_t)a * lddo + (size_t)h * HD, lddo, q0, L, tid, 128);
  load_tile_async<HD>(sO + 64 * LDS, Kg, ld, 0, L, tid, 128);
  load_tile_async<HD>(sO + 2 * 64 * LDS, Vg, ld, 0, L, tid, 128);
  cp_async_commit();
  const float c2 = scale * kLog2e;
  const int row0 = q0 + warp * 16 + (lane >> 2);
  float lrow[2], drow[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = row0 + r * 8;
    lrow[r] = row < L ? lse[(size_t)h * T + a + row] * kLog2e : 0.f;
    drow[r] = row < L ? D[(size_t)h * T + a + row] : 0.f;
  }
  float dq[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
  const int kend = min(L, q0 + 64);
  for (int k0 = 0, it = 0; k0 < kend; k0 += 64, ++it) {
    __nv_bfloat16* sK = sO + (1 + 2 * (it & 1)) * 64 * LDS;
    __nv_bfloat16* sV = sK + 64 * LDS;
    if (k0 + 64 < kend) {
      __nv_bfloat16* nK = sO + (1 + 2 * ((it + 1) & 1)) * 64 * LDS;
      load_tile_async<HD>(nK, Kg, ld, k0 + 64, L, tid, 128);
      load_tile_async<HD>(nK + 64 * LDS, Vg, ld, k0 + 64, L, tid, 128);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    float p[8][4], dp[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) p[i][e] = dp[i][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD; ks += 16) {
      uint32_t aq[4], ao[4];
      ldsm_A(aq, sQ, LDS, warp * 16, ks, lane);
      ldsm_A(ao, sO, LDS, warp * 16, ks, lane);
#pragma unroll
      for (int nt = 0; nt < 8; nt += 2) {
        uint32_t b[4];
        ldsm_B_nk(b, sK, LDS, nt * 8, ks, lane);
        mma16816(p[nt], aq, b[0], b[1]);
        mma16816(p[nt + 1], aq, b[2], b[3]);
        ldsm_B_nk(b, sV, LDS, nt * 8, ks, lane);
        mma16816(dp[nt], ao, b[0], b[1]);
        mma16816(dp[nt + 1], ao, b[2], b[3]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k0 + nt * 8 + 2 * (lane & 3) + (e & 1);
        const int row = row0 + (e >> 1) * 8;
        const float pv = (key > row || key >= L) ? 0.f : exp2f(p[nt][e] * c2 - lrow[e >> 1]);
        p[nt][e] = pv * (dp[nt][e] - drow[e >> 1]);   // dS
      }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t da[4];
      acc_to_A(da, p[2 * kk], p[2 * kk + 1]);
#pragma unroll
      for (int dn = 0; dn < HD / 8; dn += 2) {
        uint32_t b[4];
        ldsm_B_kn(b, sK, LDS, kk * 16, dn * 8, lane);
        mma16816(dq[dn], da, b[0], b[1]);
        mma16816(dq[dn + 1], da, b[2], b[3]);
      }
    }
    __syncthreads();   // every warp is done with this buffer before it is refilled
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = row0 + r * 8;
    if (row >= L) continue;
    float* grow = dqkv + (size_t)(a + row) * ldg + (size_t)h * HD;
#pragma unroll
    for (int dn = 0; dn < HD / 8; ++dn) {
      const int col = dn * 8 + 2 * (lane & 3);
      *reinterpret_cast<float2*>(grow + col) = make_float2(dq[dn][2 * r] * scale, dq[dn][2 * r + 1] * scale);
    }
  }
}

// ------------------------------------------------------------------ backward: dk, dv
// grid (ceil(maxlen / 64), nkv * hsplit, nseq).  Warp w owns keys 16w..16w+15 of the
// tile; loops over its slice of the group's query heads (all of them when hsplit = 1),
// then query tiles from the key tile on.  hsplit > 1: the slice's dk / dv go to
// part [hsplit][T][2 nkv HD] (fp32, dk already scaled) for attn_dkdv_reduce_kernel.
template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_dkdv_kernel(const __nv_bfloat16* __restrict__ qkv, long long ld,
                                                            const __nv_bfloat16* __restrict__ dout, long long lddo,
                                                            const float* __restrict__ lse,
                                                            const float* __restrict__ D, const int* __restrict__ cu,
                                                            int nh, int nkv, float scale, float* __restrict__ dqkv,
                                                            long long ldg, int T, int hsplit,
                                                            float* __restrict__ part) {
  constexpr int LDS = HD + 8;
  extern __shared__ __align__(16) uint8_t attn_smem[];
  // K, V, then two (Q, dO) buffers and two (lse, D) rows: the next query tile is copied
  // while this one computes
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(attn_smem);
  __nv_bfloat16* sV = sK + 64 * LDS;
  float* sLD = reinterpret_cast<float*>(sV + 5 * 64 * LDS);   // [2][2][64]
  const int s = blockIdx.z, g = blockIdx.y / hsplit, hs = blockIdx.y % hsplit;
  int a, L;
  seq_range(cu, s, T, a, L);
  const int k0 = blockIdx.x * 64;
  if (k0 >= L) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  load_tile_async<HD>(sK, qkv + (size_t)a * ld + (size_t)(nh + g) * HD, ld, k0, L, tid, 128);
  load_tile_async<HD>(sV, qkv + (size_t)a * ld + (size_t)(nh + nkv + g) * HD, ld, k0, L, tid, 128);
  const float c2 = scale * kLog2e;
  const int key0 = k0 + warp * 16 + (lane >> 2);
  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;
  const int group = nh / nkv;
  // this CTA's query heads: [h_lo, h_lo + nheads) of the group
  const int per = (group + hsplit - 1) / hsplit;
  const int h_lo = g * group + hs * per;
  const int nheads = max(0, min(per, group - hs * per));
  // flat loop over (query head, query tile from the key tile on)
  const int nqt = (L - k0 + 63) / 64;
  const int nit = nheads * nqt;
  auto issue = [&](int j) {
    const int h = h_lo + j / nqt, q0 = k0 + (j % nqt) * 64, buf = j & 1;
    __nv_bfloat16* dQ = sV + (1 + 2 * buf) * 64 * LDS;
    load_tile_async<HD>(dQ, qkv + (size_t)a * ld + (size_t)h * HD, ld, q0, L, tid, 128);
    load_tile_async<HD>(dQ + 64 * LDS, dout + (size_t)a * lddo + (size_t)h * HD, lddo, q0, L, tid, 128);
    if (tid < 64) {
      const int q = q0 + tid;
      sLD[buf * 128 + tid] = q < L ? lse[(size_t)h * T + a + q] * kLog2e : 0.f;
      sLD[buf * 128 + 64 + tid] = q < L ? D[(size_t)h * T + a + q] : 0.f;
    }
    cp_async_commit();
  };
  if (nit > 0) issue(0);
  else cp_async_commit();   // K / V only (no query head in this slice): nothing to wait on
  for (int j = 0; j < nit; ++j) {
    const int q0 = k0 + (j % nqt) * 64, buf = j & 1;
    const __nv_bfloat16* sQ = sV + (1 + 2 * buf) * 64 * LDS;
    const __nv_bfloat16* sO = sQ + 64 * LDS;
    const float* sL = sLD + buf * 128;
    const float* sD = sL + 64;
    {
      if (j + 1 < nit) {
        issue(j + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      float pt[8][4], dpt[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) pt[i][e] = dpt[i][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD; ks += 16) {
        uint32_t ak[4], av[4];
        ldsm_A(ak, sK, LDS, warp * 16, ks, lane);
        ldsm_A(av, sV, LDS, warp * 16, ks, lane);
#pragma unroll
        for (int nt = 0; nt < 8; nt += 2) {
          uint32_t b[4];
          ldsm_B_nk(b, sQ, LDS, nt * 8, ks, lane);
          mma16816(pt[nt], ak, b[0], b[1]);
          mma16816(pt[nt + 1], ak, b[2], b[3]);
          ldsm_B_nk(b, sO, LDS, nt * 8, ks, lane);
          mma16816(dpt[nt], av, b[0], b[1]);
          mma16816(dpt[nt + 1], av, b[2], b[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qc = nt * 8 + 2 * (lane & 3) + (e & 1);
          const int q = q0 + qc;
          const int key = key0 + (e >> 1) * 8;
          const float pv = (q < key || q >= L) ? 0.f : exp2f(pt[nt][e] * c2 - sL[qc]);
          pt[nt][e] = pv;
          dpt[nt][e] = pv * (dpt[nt][e] - sD[qc]);   // dS^T
        }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4], da[4];
        acc_to_A(pa, pt[2 * kk], pt[2 * kk + 1]);
        acc_to_A(da, dpt[2 * kk], dpt[2 * kk + 1]);
#pragma unroll
        for (int dn = 0; dn < HD / 8; dn += 2) {
          uint32_t b[4];
          ldsm_B_kn(b, sO, LDS, kk * 16, dn * 8, lane);
          mma16816(dv[dn], pa, b[0], b[1]);
          mma16816(dv[dn + 1], pa, b[2], b[3]);
          ldsm_B_kn(b, sQ, LDS, kk * 16, dn * 8, lane);
          mma16816(dk[dn], da, b[0], b[1]);
          mma16816(dk[dn + 1], da, b[2], b[3]);
        }
      }
      __syncthreads();   // every warp is done with this buffer before it is refilled
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int key = key0 + r * 8;
    if (key >= L) continue;
    float* krow = hsplit > 1 ? part + ((size_t)hs * T + a + key) * (2 * nkv * HD) + (size_t)g * HD
                             : dqkv + (size_t)(a + key) * ldg + (size_t)(nh + g) * HD;
    float* vrow = hsplit > 1 ? krow + (size_t)nkv * HD : dqkv + (size_t)(a + key) * ldg + (size_t)(nh + nkv + g) * HD;
#pragma unroll
    for (int dn = 0; dn < HD / 8; ++dn) {
      const int col = dn * 8 + 2 * (lane & 3);
      *reinterpret_cast<float2*>(krow + col) = make_float2(dk[dn][2 * r] * scale, dk[dn][2 * r + 1] * scale);
      *reinterpret_cast<float2*>(vrow + col) = make_float2(dv[dn][2 * r], dv[dn][2 * r + 1]);
    }
  }
}

// dk / dv = sum over the head slices in slice order, into the k / v columns of dqkv.
// Four consecutive columns per thread (float4): w = 2 nkv hd and ldg are multiples of 4.
__global__ void attn_dkdv_reduce_kernel(const float* __restrict__ part, int hsplit, int nh, int nkv, int hd, int T,
                                        float* __restrict__ dqkv, long long ldg) {
  const long long w4 = (2LL * nkv * hd) >> 2;
  const long long n4 = (long long)T * w4;
  const float4* p4 = reinterpret_cast<const float4*>(part);
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n4; e += (long long)gridDim.x * blockDim.x) {
    const long long t = e / w4, c = (e % w4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < hsplit; ++k) {
      const float4 x = p4[(size_t)k * n4 + e];
      v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
    }
    *reinterpret_cast<float4*>(dqkv + t * ldg + (long long)nh * hd + c) = v;
  }
}

}  // namespace ls
