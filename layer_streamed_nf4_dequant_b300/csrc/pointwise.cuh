// Bandwidth-bound kernels of the decoder layer and the loss: RMSNorm, RoPE, SwiGLU,
// NF4 embedding gather, next-token targets, vocabulary log-sum-exp combine,
// per-sequence logprob sums, the DPO loss, and the LoRA low-rank pieces.
//
// Rows are handled one warp each with 16-byte vector accesses; every reduction has
// a fixed order (lane-strided partials, then a butterfly), so results do not depend
// on scheduling and a streamed run repeats a resident one bit for bit.
#pragma once
#include "common.cuh"

namespace ls {

// ------------------------------------------------------------------ bounded waits
// One thread waits, through the same bounded loop as the split GEMM's partial-tile
// exchange, until *flag == value or limit_ns has passed; status 0 = seen, 1 = ran out.
__global__ void wait_flag_kernel(const unsigned* flag, unsigned value, unsigned long long limit_ns, int* status) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  *status = flag_wait_eq(flag, value, limit_ns) ? 0 : 1;
}

// ------------------------------------------------------------------ RMSNorm
// y = bf16(w * bf16(x * rstd)), rstd = 1 / sqrt(mean(x^2) + eps)   (x bf16 [T, H])
__global__ void rmsnorm_fwd_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
                                   __nv_bfloat16* __restrict__ y, float* __restrict__ rstd, int T, int H,
                                   float eps) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * H);
  const int nv = H >> 3;
  float ss = 0.f;
  for (int v = lane; v < nv; v += 32) {
    const uint4 p = xr[v];
    const uint32_t q[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16lo(q[e]), b = bf16hi(q[e]);
      ss += a * a;
      ss += b * b;
    }
  }
  ss = warp_sum(ss);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
  if (lane == 0 && rstd) rstd[row] = r;
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * H);
  for (int v = lane; v < nv; v += 32) {
    const uint4 p = xr[v], wv = wr[v];
    const uint32_t q[4] = {p.x, p.y, p.z, p.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float n0 = __bfloat162float(__float2bfloat16_rn(bf16lo(q[e]) * r));
      const float n1 = __bfloat162float(__float2bfloat16_rn(bf16hi(q[e]) * r));
      o[e] = pack_bf16x2(bf16lo(ww[e]) * n0, bf16hi(ww[e]) * n1);
    }
    yr[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// dx += rstd * (g - n * mean(g * n)),  g = dy * w,  n = x * rstd.   dx fp32, and an
// optional bf16 copy of the updated dx (the next matrix product's input).
__global__ void rmsnorm_bwd_kernel(const float* __restrict__ dy, const __nv_bfloat16* __restrict__ x,
                                   const float* __restrict__ rstd, const __nv_bfloat16* __restrict__ w,
                                   float* __restrict__ dx, __nv_bfloat16* __restrict__ dx_bf16, int T, int H,
                                   int accumulate) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const float r = rstd[row];
  const int nv = H >> 2;
  const float4* dyr = reinterpret_cast<const float4*>(dy + (size_t)row * H);
  const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)row * H);
  const uint2* wr = reinterpret_cast<const uint2*>(w);
  float dot = 0.f;
  for (int v = lane; v < nv; v += 32) {
    const float4 d = dyr[v];
    const uint2 xv = xr[v], wv = wr[v];
    dot += d.x * bf16lo(wv.x) * (bf16lo(xv.x) * r);
    dot += d.y * bf16hi(wv.x) * (bf16hi(xv.x) * r);
    dot += d.z * bf16lo(wv.y) * (bf16lo(xv.y) * r);
    dot += d.w * bf16hi(wv.y) * (bf16hi(xv.y) * r);
  }
  dot = warp_sum(dot);
  const float c = dot / (float)H;
  float4* dxr = reinterpret_cast<float4*>(dx + (size_t)row * H);
  uint2* db = dx_bf16 ? reinterpret_cast<uint2*>(dx_bf16 + (size_t)row * H) : nullptr;
  for (int v = lane; v < nv; v += 32) {
    const float4 d = dyr[v];
    const uint2 xv = xr[v], wv = wr[v];
    float4 o = accumulate ? dxr[v] : make_float4(0.f, 0.f, 0.f, 0.f);
    o.x += r * (d.x * bf16lo(wv.x) - bf16lo(xv.x) * r * c);
    o.y += r * (d.y * bf16hi(wv.x) - bf16hi(xv.x) * r * c);
    o.z += r * (d.z * bf16lo(wv.y) - bf16lo(xv.y) * r * c);
    o.w += r * (d.w * bf16hi(wv.y) - bf16hi(xv.y) * r * c);
    dxr[v] = o;
    if (db) db[v] = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
  }
}

// Row-per-block forms of the two RMSNorm kernels above (same formulas).  With one warp
// per row, T = 1024 rows put only 7 warps on an SM; here a block of 4 (forward) or 8
// (backward) warps takes one row and keeps its slice of the row in registers, so x and
// dy are read from memory once and every SM has tens of warps in flight.  Thread i
// holds the 16-byte (forward: 8 bf16) or float4 (backward) chunks i, i + blockDim, ...
// (VPT of them, guarded by the row length); the sums run per thread in chunk order, then
// a warp butterfly, then the warps in order: fixed, so results do not depend on
// scheduling.
__device__ __forceinline__ float block_sum_ordered(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

template <int VPT>
__global__ void __launch_bounds__(128) rmsnorm_fwd_row_kernel(const __nv_bfloat16* __restrict__ x,
                                                              const __nv_bfloat16* __restrict__ w,
                                                              __nv_bfloat16* __restrict__ y, float* __restrict__ rstd,
                                                              int H, float eps) {
  __shared__ float red[4];
  const int row = blockIdx.x;
  const int nv = H >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * H);
  uint4 xv[VPT];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * 128;
    xv[i] = v < nv ? xr[v] : make_uint4(0, 0, 0, 0);
    const uint32_t q[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16lo(q[e]), b = bf16hi(q[e]);
      ss += a * a;
      ss += b * b;
    }
  }
  ss = block_sum_ordered(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)H + eps);
  if (threadIdx.x == 0 && rstd) rstd[row] = r;
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * H);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * 128;
    if (v >= nv) continue;
    const uint4 wv = wr[v];
    const uint32_t q[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float n0 = __bfloat162float(__float2bfloat16_rn(bf16lo(q[e]) * r));
      const float n1 = __bfloat162float(__float2bfloat16_rn(bf16hi(q[e]) * r));
      o[e] = pack_bf16x2(bf16lo(ww[e]) * n0, bf16hi(ww[e]) * n1);
    }
    yr[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int VPT>
__global__ void __launch_bounds__(256) rmsnorm_bwd_row_kernel(const float* __restrict__ dy,
                                                              const __nv_bfloat16* __restrict__ x,
                                                              const float* __restrict__ rstd,
                                                              const __nv_bfloat16* __restrict__ w,
                                                              float* __restrict__ dx, __nv_bfloat16* __restrict__ dx_bf16,
                                                              int H, int accumulate) {
  __shared__ float red[8];
  const int row = blockIdx.x;
  const float r = rstd[row];
  const int nv = H >> 2;
  const float4* dyr = reinterpret_cast<const float4*>(dy + (size_t)row * H);
  const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)row * H);
  const uint2* wr = reinterpret_cast<const uint2*>(w);
  float4 d[VPT];
  uint2 xv[VPT], wv[VPT];
  float dot = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * 256;
    const bool ok = v < nv;
    d[i] = ok ? dyr[v] : make_float4(0.f, 0.f, 0.f, 0.f);
    xv[i] = ok ? xr[v] : make_uint2(0, 0);
    wv[i] = ok ? wr[v] : make_uint2(0, 0);
    dot += d[i].x * bf16lo(wv[i].x) * (bf16lo(xv[i].x) * r);
    dot += d[i].y * bf16hi(wv[i].x) * (bf16hi(xv[i].x) * r);
    dot += d[i].z * bf16lo(wv[i].y) * (bf16lo(xv[i].y) * r);
    dot += d[i].w * bf16hi(wv[i].y) * (bf16hi(xv[i].y) * r);
  }
  const float c = block_sum_ordered(dot, red) / (float)H;
  float4* dxr = reinterpret_cast<float4*>(dx + (size_t)row * H);
  uint2* db = dx_bf16 ? reinterpret_cast<uint2*>(dx_bf16 + (size_t)row * H) : nullptr;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * 256;
    if (v >= nv) continue;
    float4 o = accumulate ? dxr[v] : make_float4(0.f, 0.f, 0.f, 0.f);
    o.x += r * (d[i].x * bf16lo(wv[i].x) - bf16lo(xv[i].x) * r * c);
    o.y += r * (d[i].y * bf16hi(wv[i].x) - bf16hi(xv[i].x) * r * c);
    o.z += r * (d[i].z * bf16lo(wv[i].y) - bf16lo(xv[i].y) * r * c);
    o.w += r * (d[i].w * bf16hi(wv[i].y) - bf16hi(xv[i].y) * r * c);
    dxr[v] = o;
    if (db) db[v] = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
  }
}

// ------------------------------------------------------------------ RoPE
// In place on the q and k heads of qkv [T, ld] (bf16): pair (i, i + hd/2) turned by
// the angle pos * theta^(-2i/hd); cos/sin come from a [max_pos, hd/2] fp32 table.
__global__ void rope_fwd_kernel(__nv_bfloat16* __restrict__ qkv, long long ld, const int* __restrict__ pos,
                                const float* __restrict__ cs, const float* __restrict__ sn, int T, int nheads,
                                int hd) {
  const int half = hd >> 1;
  const long long total = (long long)T * nheads * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(idx % half);
    const long long th = idx / half;
    const int h = (int)(th % nheads);
    const int t = (int)(th / nheads);
    __nv_bfloat16* p = qkv + (size_t)t * ld + (size_t)h * hd;
    const int ps = pos[t];
    const float c = cs[(size_t)ps * half + i], s = sn[(size_t)ps * half + i];
    const float x1 = bf2f(p[i]), x2 = bf2f(p[i + half]);
    p[i] = __float2bfloat16_rn(x1 * c - x2 * s);
    p[i + half] = __float2bfloat16_rn(x2 * c + x1 * s);
  }
}

// Backward of RoPE (rotation by -angle) on the q and k columns of an fp32 gradient,
// written as bf16 together with the untouched v columns: dqkv = bf16(R^T dqkv_f).
__global__ void rope_bwd_cast_kernel(const float* __restrict__ g, __nv_bfloat16* __restrict__ out, long long ld,
                                     const int* __restrict__ pos, const float* __restrict__ cs,
                                     const float* __restrict__ sn, int T, int nrot_heads, int hd, int ncols) {
  const int half = hd >> 1;
  const int rot_cols = nrot_heads * hd;
  const long long total = (long long)T * ncols;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int col = (int)(idx % ncols);
    const int t = (int)(idx / ncols);
    const float* gr = g + (size_t)t * ld;
    float v;
    if (col < rot_cols) {
      const int i = col % hd, base = col - i;
      const int ii = i < half ? i : i - half;
      const int ps = pos[t];
      const float c = cs[(size_t)ps * half + ii], s = sn[(size_t)ps * half + ii];
      const float y1 = gr[base + ii], y2 = gr[base + ii + half];
      v = i < half ? (y1 * c + y2 * s) : (y2 * c - y1 * s);
    } else {
      v = gr[col];
    }
    out[(size_t)t * ld + col] = __float2bfloat16_rn(v);
  }
}

// 16-byte forms of the two RoPE kernels (same arithmetic, element for element): a
// thread turns 8 consecutive pairs (i .. i+7, i+hd/2 .. i+hd/2+7) of one head, with
// 16-byte loads and stores of q/k and 2 x float4 table reads.  hd/2 must be a multiple
// of 8 (hd 64 and 128 are).
__global__ void rope_fwd_vec_kernel(__nv_bfloat16* __restrict__ qkv, long long ld, const int* __restrict__ pos,
                                    const float* __restrict__ cs, const float* __restrict__ sn, int T, int nheads,
                                    int hd) {
  const int half = hd >> 1, g8 = half >> 3;
  const long long total = (long long)T * nheads * g8;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int i0 = (int)(idx % g8) * 8;
    const long long th = idx / g8;
    const int h = (int)(th % nheads);
    const int t = (int)(th / nheads);
    __nv_bfloat16* p = qkv + (size_t)t * ld + (size_t)h * hd;
    const size_t tb = (size_t)pos[t] * half + i0;
    const float4 c0 = *reinterpret_cast<const float4*>(cs + tb), c1 = *reinterpret_cast<const float4*>(cs + tb + 4);
    const float4 s0 = *reinterpret_cast<const float4*>(sn + tb), s1 = *reinterpret_cast<const float4*>(sn + tb + 4);
    const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const uint4 a = *reinterpret_cast<const uint4*>(p + i0), b = *reinterpret_cast<const uint4*>(p + i0 + half);
    const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x1l = bf16lo(aa[e]), x1h = bf16hi(aa[e]), x2l = bf16lo(bb[e]), x2h = bf16hi(bb[e]);
      const int k = 2 * e;
      oa[e] = pack_bf16x2(x1l * c[k] - x2l * sv[k], x1h * c[k + 1] - x2h * sv[k + 1]);
      ob[e] = pack_bf16x2(x2l * c[k] + x1l * sv[k], x2h * c[k + 1] + x1h * sv[k + 1]);
    }
    *reinterpret_cast<uint4*>(p + i0) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *reinterpret_cast<uint4*>(p + i0 + half) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// Backward: a thread takes 4 consecutive pairs of one rotated head (float4 reads of
// both halves, two 8-byte bf16 stores), or 8 consecutive unrotated columns.
__global__ void rope_bwd_cast_vec_kernel(const float* __restrict__ g, __nv_bfloat16* __restrict__ out, long long ld,
                                         const int* __restrict__ pos, const float* __restrict__ cs,
                                         const float* __restrict__ sn, int T, int nrot_heads, int hd, int ncols) {
  const int half = hd >> 1;
  const int rot_units = nrot_heads * (half >> 2);        // 4-pair units of the rotated heads
  const int plain_units = (ncols - nrot_heads * hd) >> 3;  // 8-column units of the rest
  const int units = rot_units + plain_units;
  const long long total = (long long)T * units;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int u = (int)(idx % units);
    const int t = (int)(idx / units);
    const float* gr = g + (size_t)t * ld;
    __nv_bfloat16* orow = out + (size_t)t * ld;
    if (u < rot_units) {
      const int h = u / (half >> 2), i0 = (u % (half >> 2)) * 4;
      const int base = h * hd;
      const size_t tb = (size_t)pos[t] * half + i0;
      const float4 c = *reinterpret_cast<const float4*>(cs + tb), s = *reinterpret_cast<const float4*>(sn + tb);
      const float4 y1 = *reinterpret_cast<const float4*>(gr + base + i0);
      const float4 y2 = *reinterpret_cast<const float4*>(gr + base + i0 + half);
      *reinterpret_cast<uint2*>(orow + base + i0) =
          make_uint2(pack_bf16x2(y1.x * c.x + y2.x * s.x, y1.y * c.y + y2.y * s.y),
                     pack_bf16x2(y1.z * c.z + y2.z * s.z, y1.w * c.w + y2.w * s.w));
      *reinterpret_cast<uint2*>(orow + base + i0 + half) =
          make_uint2(pack_bf16x2(y2.x * c.x - y1.x * s.x, y2.y * c.y - y1.y * s.y),
                     pack_bf16x2(y2.z * c.z - y1.z * s.z, y2.w * c.w - y1.w * s.w));
    } else {
      const int col = nrot_heads * hd + (u - rot_units) * 8;
      const float4 a = *reinterpret_cast<const float4*>(gr + col), b = *reinterpret_cast<const float4*>(gr + col + 4);
      *reinterpret_cast<uint4*>(orow + col) = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                                         pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
  }
}

// ------------------------------------------------------------------ SwiGLU
// gu [T, 2I] = [gate | up] (bf16)  ->  h [T, I] = bf16(silu(gate) * up)
__global__ void swiglu_fwd_kernel(const __nv_bfloat16* __restrict__ gu, __nv_bfloat16* __restrict__ h, int T,
                                  int I) {
  const long long n8 = (long long)T * (I >> 3);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n8;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / (I >> 3)), c = (int)(idx % (I >> 3));
    const uint4 gv = reinterpret_cast<const uint4*>(gu + (size_t)t * 2 * I)[c];
    const uint4 uv = reinterpret_cast<const uint4*>(gu + (size_t)t * 2 * I + I)[c];
    const uint32_t ga[4] = {gv.x, gv.y, gv.z, gv.w}, ua[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float g0 = bf16lo(ga[e]), g1 = bf16hi(ga[e]);
      const float s0 = g0 / (1.f + __expf(-g0)), s1 = g1 / (1.f + __expf(-g1));
      o[e] = pack_bf16x2(s0 * bf16lo(ua[e]), s1 * bf16hi(ua[e]));
    }
    reinterpret_cast<uint4*>(h + (size_t)t * I)[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// dh fp32 [T, I]  ->  dgu [T, 2I] bf16:  d gate = dh * up * silu'(gate),  d up = dh * silu(gate)
__global__ void swiglu_bwd_kernel(const float* __restrict__ dh, const __nv_bfloat16* __restrict__ gu,
                                  __nv_bfloat16* __restrict__ dgu, int T, int I) {
  const long long n4 = (long long)T * (I >> 2);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n4;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / (I >> 2)), c = (int)(idx % (I >> 2));
    const float4 d = reinterpret_cast<const float4*>(dh + (size_t)t * I)[c];
    const uint2 gv = reinterpret_cast<const uint2*>(gu + (size_t)t * 2 * I)[c];
    const uint2 uv = reinterpret_cast<const uint2*>(gu + (size_t)t * 2 * I + I)[c];
    const float dd[4] = {d.x, d.y, d.z, d.w};
    const float g[4] = {bf16lo(gv.x), bf16hi(gv.x), bf16lo(gv.y), bf16hi(gv.y)};
    const float u[4] = {bf16lo(uv.x), bf16hi(uv.x), bf16lo(uv.y), bf16hi(uv.y)};
    float dg[4], du[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float sg = 1.f / (1.f + __expf(-g[e]));
      const float silu = g[e] * sg;
      dg[e] = dd[e] * u[e] * (sg * (1.f + g[e] * (1.f - sg)));
      du[e] = dd[e] * silu;
    }
    reinterpret_cast<uint2*>(dgu + (size_t)t * 2 * I)[c] = make_uint2(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]));
    reinterpret_cast<uint2*>(dgu + (size_t)t * 2 * I + I)[c] = make_uint2(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]));
  }
}

// ------------------------------------------------------------------ embedding
// x[t] = dequant(row tokens[t] of the NF4 embedding); packed/absmax may live in
// mapped pinned host memory (only the T selected rows cross the host link).
// A token id outside [0, V) gives a zero row and raises the device error word (the
// table may be mapped host memory: an unchecked id would read outside the mapping).
__global__ void embed_gather_kernel(const int* __restrict__ tokens, const uint8_t* __restrict__ packed,
                                    const float* __restrict__ absmax, __nv_bfloat16* __restrict__ x, int T,
                                    int H, int V) {
  const int nch = H >> 3;   // 8-element chunks per row
  const long long total = (long long)T * nch;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / nch), c = (int)(idx % nch);
    const long long tok = tokens[t];
    if (tok < 0 || tok >= V) {
      if (c == 0) raise_error(DEV_BAD_ARG);
      reinterpret_cast<uint4*>(x + (size_t)t * H)[c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint32_t w = *reinterpret_cast<const uint32_t*>(packed + tok * (H >> 1) + c * 4);
    const float a = absmax[tok * (H >> 6) + (c >> 3)];
    uint32_t o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
      o[b] = pack_bf16x2(kNF4Table[(w >> (8 * b + 4)) & 15] * a, kNF4Table[(w >> (8 * b)) & 15] * a);
    reinterpret_cast<uint4*>(x + (size_t)t * H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Plain NF4 dequantisation of a whole matrix (rows x cols) to bf16.
__global__ void nf4_dequant_kernel(const uint8_t* __restrict__ packed, const float* __restrict__ absmax,
                                   __nv_bfloat16* __restrict__ out, long long rows, int cols) {
  const int nch = cols >> 3;
  const long long total = rows * nch;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long r = idx / nch;
    const int c = (int)(idx % nch);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(packed + r * (cols >> 1) + c * 4);
    const float a = absmax[r * (cols >> 6) + (c >> 3)];
    uint32_t o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
      o[b] = pack_bf16x2(kNF4Table[(w >> (8 * b + 4)) & 15] * a, kNF4Table[(w >> (8 * b)) & 15] * a);
    reinterpret_cast<uint4*>(out + r * cols)[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------ sequences
// Per position: position within its sequence, next-token target (-1 at a sequence's
// last position), and the loss coefficient seq_coef[seq] * mask (when given).
__global__ void seq_setup_kernel(const int* __restrict__ tokens, const int* __restrict__ cu, int nseq,
                                 const uint8_t* __restrict__ mask, const float* __restrict__ seq_coef,
                                 int* __restrict__ pos, int* __restrict__ tgt, float* __restrict__ coef, int T) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int s = 0;
  while (s + 1 < nseq && cu[s + 1] <= t) ++s;
  const int a = cu[s], b = cu[s + 1];
  if (pos) pos[t] = t - a;
  if (tgt) tgt[t] = (t + 1 < b && t + 1 < T) ? tokens[t + 1] : -1;
  if (coef) coef[t] = (seq_coef && mask && mask[t] && t + 1 < b) ? seq_coef[s] : 0.f;
}

// Doubled batch of the shared-read DPO forward: tok2 = [tok; tok] and sequence offsets
// cu2 = [cu; T + cu[1..nseq]] (the reference copy of every sequence follows the policy copies).
__global__ void pair_setup_kernel(const int* __restrict__ tokens, const int* __restrict__ cu, int nseq, int T,
                                  int* __restrict__ tok2, int* __restrict__ cu2) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 2 * T) tok2[i] = tokens[i < T ? i : i - T];
  if (i <= 2 * nseq) cu2[i] = i <= nseq ? cu[i] : T + cu[i - nseq];
}

// lse[t] = log sum_v exp(logit) from per-column-group (max, sum-exp) partials, in
// partial order; lp[t] = logit[t, target] - lse[t] (0 without a target).  Two passes
// over the row's partials (max, then the rescaled sum): every load of a pass is
// independent, and each partial costs one exp.
__global__ void logprob_combine_kernel(const float* __restrict__ pmax, const float* __restrict__ psum, int P,
                                       int ld, const float* __restrict__ tgt_logit, const int* __restrict__ tgt,
                                       float* __restrict__ lse, float* __restrict__ lp, int T) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= T) return;
  const float* pm = pmax + (size_t)row * ld;
  const float* ps = psum + (size_t)row * ld;
  float m = -INFINITY;
  for (int p = lane; p < P; p += 32) m = fmaxf(m, pm[p]);
  m = warp_max(m);
  float s = 0.f;
  for (int p = lane; p < P; p += 32) s += ps[p] * __expf(pm[p] - m);
  s = warp_sum(s);
  if (lane == 0) {
    const float l = m + logf(s);
    lse[row] = l;
    lp[row] = tgt[row] >= 0 ? tgt_logit[row] - l : 0.f;
  }
}

// sums[s] = sum over positions t of sequence s of mask[t] * lp[t] (one block per sequence)
__global__ void seq_sum_kernel(const float* __restrict__ lp, const uint8_t* __restrict__ mask,
                               const int* __restrict__ cu, float* __restrict__ sums) {
  const int s = blockIdx.x;
  const int a = cu[s], b = cu[s + 1];
  float acc = 0.f;
  for (int t = a + threadIdx.x; t < b; t += blockDim.x) acc += mask[t] ? lp[t] : 0.f;
  __shared__ float red[32];
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) sums[s] = v;
  }
}

// DPO: z_p = beta ((pi_c - ref_c) - (pi_r - ref_r)), loss = mean_p softplus(-z_p);
// coeffs = dL/d(sequence logprob sum): chosen -beta sigma(-z)/P, rejected +beta sigma(-z)/P.
__global__ void dpo_loss_kernel(const float* __restrict__ pi, const float* __restrict__ ref, int npairs,
                                float beta, float* __restrict__ loss, float* __restrict__ coeffs) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  float acc = 0.f;
  for (int p = 0; p < npairs; ++p) {
    const float z = beta * ((pi[2 * p] - ref[2 * p]) - (pi[2 * p + 1] - ref[2 * p + 1]));
    const float nz = -z;
    acc += fmaxf(nz, 0.f) + log1pf(__expf(-fabsf(nz)));   // softplus(-z), stable
    const float sig = 1.f / (1.f + __expf(z));            // sigma(-z)
    if (coeffs) {
      coeffs[2 * p] = -beta * sig / (float)npairs;
      coeffs[2 * p + 1] = beta * sig / (float)npairs;
    }
  }
  if (loss) *loss = acc / (float)npairs;
}

// Other preference losses over (chosen, rejected) pairs or labelled sequences, from
// per-sequence logprob sums (the pages list ORPO, SimPO and KTO beside DPO; the formulas
// are the methods' own).  One block: the response lengths |y| come from the loss mask
// (a fixed-order block reduction per sequence), then thread 0 forms the loss and each
// sequence's coefficient dL/d(sum) for the streamed backward.
enum PrefKind : int { PREF_SIMPO = 0, PREF_ORPO = 1, PREF_KTO = 2 };

__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x))); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + __expf(-x)); }

__global__ void pref_loss_kernel(int kind, const float* __restrict__ pi, const float* __restrict__ ref,
                                 const int* __restrict__ cu, const uint8_t* __restrict__ mask,
                                 const uint8_t* __restrict__ desirable, int nseq, float beta, float p1, float p2,
                                 float* __restrict__ loss, float* __restrict__ coeffs) {
  extern __shared__ float cnt[];   // [nseq]
  __shared__ float red[32];
  if (kind != PREF_KTO) {
    for (int sq = 0; sq < nseq; ++sq) {
      const int a = cu[sq], b = cu[sq + 1];
      float c = 0.f;
      for (int t = a + threadIdx.x; t < b; t += blockDim.x) c += mask[t] ? 1.f : 0.f;
      c = warp_sum(c);
      if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
      __syncthreads();
      if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) cnt[sq] = v;
      }
      __syncthreads();
    }
  }
  if (threadIdx.x != 0) return;
  float acc = 0.f;
  if (kind == PREF_SIMPO || kind == PREF_ORPO) {
    const int np = nseq / 2;
    for (int p = 0; p < np; ++p) {
      const float nc = cnt[2 * p], nr = cnt[2 * p + 1];
      const float lc = pi[2 * p] / nc, lr = pi[2 * p + 1] / nr;
      if (kind == PREF_SIMPO) {   // p1 = gamma
        const float z = beta * (lc - lr) - p1;
        acc += softplus_f(-z);
        const float sg = sigmoid_f(-z);
        if (coeffs) {
          coeffs[2 * p] = -sg * beta / nc / (float)np;
          coeffs[2 * p + 1] = sg * beta / nr / (float)np;
        }
      } else {                    // p1 = lambda; log odds = l - log(1 - e^l)
        const float emc = expm1f(lc), emr = expm1f(lr);
        const float d = (lc - logf(-emc)) - (lr - logf(-emr));
        acc += -lc + p1 * softplus_f(-d);
        const float sg = sigmoid_f(-d);
        if (coeffs) {             // d log odds / d l = -1 / expm1(l)
          coeffs[2 * p] = (-1.f + p1 * sg / emc) / nc / (float)np;
          coeffs[2 * p + 1] = (-p1 * sg / emr) / nr / (float)np;
        }
      }
    }
    if (loss) *loss = acc / (float)np;
  } else {                        // KTO: p1 = lambda_d, p2 = lambda_u
    float z0 = 0.f;
    for (int sq = 0; sq < nseq; ++sq) z0 += pi[sq] - ref[sq];
    z0 = fmaxf(z0 / (float)nseq, 0.f);
    for (int sq = 0; sq < nseq; ++sq) {
      const float r = pi[sq] - ref[sq];
      const bool des = desirable ? desirable[sq] != 0 : (sq % 2 == 0);
      const float lam = des ? p1 : p2;
      const float sg = sigmoid_f(beta * (des ? r - z0 : z0 - r));
      acc += lam * (1.f - sg);
      if (coeffs) coeffs[sq] = (des ? -1.f : 1.f) * lam * beta * sg * (1.f - sg) / (float)nseq;
    }
    if (loss) *loss = acc / (float)nseq;
  }
}

// ------------------------------------------------------------------ optimizer
// AdamW on the four adapter tensors of one layer (A_q, B_q, A_v, B_v), in place:
// fp32 master / first / second moments at flat offsets, bf16 copy for the forward,
// optional zeroing of the gradient.  bc1 = 1 - beta1^t, bc2 = 1 - beta2^t.
struct AdamLayer {
  float* g[4];
  __nv_bfloat16* p[4];
  long long off[4], n[4];
};

__global__ void adamw_layer_kernel(AdamLayer L, float* __restrict__ master, float* __restrict__ m1,
                                   float* __restrict__ m2, float lr, float beta1, float beta2, float eps, float wd,
                                   float bc1, float bc2, int zero_grads) {
  const int tsel = blockIdx.y;
  const long long n = L.n[tsel];
  float* g = L.g[tsel];
  __nv_bfloat16* p = L.p[tsel];
  const long long off = L.off[tsel];
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float gi = g[i];
    float w = master[off + i] * (1.f - lr * wd);
    const float a = beta1 * m1[off + i] + (1.f - beta1) * gi;
    const float b = beta2 * m2[off + i] + (1.f - beta2) * gi * gi;
    w -= lr * (a / bc1) / (sqrtf(b / bc2) + eps);
    master[off + i] = w;
    m1[off + i] = a;
    m2[off + i] = b;
    p[i] = __float2bfloat16_rn(w);
    if (zero_grads) g[i] = 0.f;
  }
}

// fp32 copy of one bf16 tensor (the optimizer's master weights at start).
__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ in, float* __restrict__ out, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    out[i] = __bfloat162float(in[i]);
}

// ------------------------------------------------------------------ LoRA pieces
// Rank-r projections of the LoRA branch (Soup's soup.yaml listing: r 16 on q_proj and
// v_proj), as one small contraction with N = 2 x 16 output columns:
//   out[t, 16 h + j] = sum_k X[t, xcol_h + k] * W_h[j, k]      (h = 0, 1; j < r, else 0)
// Forward down-projection: X = normed input, W_h = A_q / A_v  [r, K]   (row-major)
// Backward du:             X = dY (q / v columns), W_h = B_q^T / B_v^T (B [N, r], read transposed)
// Results: out_f32 [T, 32] = s * sum (optional) and out_ext [T, 64] = bf16(s * sum) with
// columns 32..63 zero (the extra reduction stage of the fused NF4 GEMM).
// Tensor cores through mma.sync m16n8k16 (bf16 in, fp32 accumulate).  One block = 16
// rows; its 8 warps split K evenly and are summed in warp order, so the result does not
// depend on scheduling.
struct LoraProjHalf {
  const __nv_bfloat16* w;   // null: this half is absent (columns stay zero)
  long long ldw;            // row pitch of W_h when not transposed
  int xcol, K, trans;
};

__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lora_w_pair(const LoraProjHalf& h, int n, int k, int r) {
  if (n >= r) return 0u;
  if (!h.trans) return *reinterpret_cast<const uint32_t*>(h.w + (size_t)n * h.ldw + k);
  const uint16_t* w = reinterpret_cast<const uint16_t*>(h.w);
  return (uint32_t)w[(size_t)k * r + n] | ((uint32_t)w[(size_t)(k + 1) * r + n] << 16);
}

// blockIdx.y / gridDim.y selects a slice of K (fixed split); with gridDim.y > 1 the
// block writes its unscaled partial sums to part [gridDim.y][T][32] for
// lora_proj_reduce_kernel instead of the outputs.
// V16: rows are read 16 bytes per lane (X and W 16-byte aligned, ldx, ldw and the column
// offsets multiples of 8, K a multiple of 32): lane (g, q) loads columns 8q .. 8q+7 of a 32-wide
// step for rows g and g + 8, and the two m16n8k16 MMAs of the step take them as their
// k positions in the order (8q, 8q+1 | 8q+2, 8q+3) and (8q+4, 8q+5 | 8q+6, 8q+7); B is
// read with the same assignment (for a row-major W, one 16-byte read of row n), so each
// MMA still sums matching X and W columns.
template <bool V16>
__global__ void __launch_bounds__(256) lora_proj_kernel(const __nv_bfloat16* __restrict__ X, long long ldx, int T,
                                                        LoraProjHalf h0, LoraProjHalf h1, int r, float s,
                                                        float* __restrict__ out_f32,
                                                        __nv_bfloat16* __restrict__ out_ext,
                                                        float* __restrict__ part) {
  __shared__ float red[8][16][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, cq = lane & 3;
  const int r0 = blockIdx.x * 16;
  const int nsplit = gridDim.y, split = blockIdx.y;
  const bool ok0 = r0 + g < T, ok1 = r0 + g + 8 < T;
  const __nv_bfloat16* x0 = X + (size_t)(ok0 ? r0 + g : 0) * ldx;
  const __nv_bfloat16* x1 = X + (size_t)(ok1 ? r0 + g + 8 : 0) * ldx;
  float acc[2][2][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) (&acc[0][0][0])[i] = 0.f;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const LoraProjHalf& h = hh ? h1 : h0;
    if (!h.w) continue;
    if constexpr (V16) {
      const int ksteps = h.K >> 5;
      const int wper = (ksteps + nsplit * 8 - 1) / (nsplit * 8);   // 32-wide k-steps per warp
      const int kb = (split * 8 + warp) * wper, ke = min(ksteps, kb + wper);
#pragma unroll 2
      for (int ks = kb; ks < ke; ++ks) {
        const int kc = (ks << 5) + 8 * cq;
        const int xc = h.xcol + kc;
        const uint4 A0 = ok0 ? *reinterpret_cast<const uint4*>(x0 + xc) : make_uint4(0, 0, 0, 0);
        const uint4 A1 = ok1 ? *reinterpret_cast<const uint4*>(x1 + xc) : make_uint4(0, 0, 0, 0);
        const uint32_t a0[4] = {A0.x, A1.x, A0.y, A1.y}, a1[4] = {A0.z, A1.z, A0.w, A1.w};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int n = nt * 8 + g;
          if (!h.trans) {   // W row n, columns kc .. kc+7: one 16-byte read for both MMAs
            const uint4 b = n < r ? *reinterpret_cast<const uint4*>(h.w + (size_t)n * h.ldw + kc) : make_uint4(0, 0, 0, 0);
            mma_16816_bf16(acc[hh][nt], a0, b.x, b.y);
            mma_16816_bf16(acc[hh][nt], a1, b.z, b.w);
          } else {
            mma_16816_bf16(acc[hh][nt], a0, lora_w_pair(h, n, kc, r), lora_w_pair(h, n, kc + 2, r));
            mma_16816_bf16(acc[hh][nt], a1, lora_w_pair(h, n, kc + 4, r), lora_w_pair(h, n, kc + 6, r));
          }
        }
      }
    } else {
      const int ksteps = h.K >> 4;
      const int wper = (ksteps + nsplit * 8 - 1) / (nsplit * 8);   // k-steps per warp
      const int kb = (split * 8 + warp) * wper, ke = min(ksteps, kb + wper);
#pragma unroll 4
      for (int ks = kb; ks < ke; ++ks) {
        const int k0 = ks << 4;
        const int xc = h.xcol + k0 + 2 * cq;
        uint32_t a[4];
        a[0] = ok0 ? *reinterpret_cast<const uint32_t*>(x0 + xc) : 0u;
        a[1] = ok1 ? *reinterpret_cast<const uint32_t*>(x1 + xc) : 0u;
        a[2] = ok0 ? *reinterpret_cast<const uint32_t*>(x0 + xc + 8) : 0u;
        a[3] = ok1 ? *reinterpret_cast<const uint32_t*>(x1 + xc + 8) : 0u;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int n = nt * 8 + g;
          const uint32_t b0 = lora_w_pair(h, n, k0 + 2 * cq, r);
          const uint32_t b1 = lora_w_pair(h, n, k0 + 8 + 2 * cq, r);
          mma_16816_bf16(acc[hh][nt], a, b0, b1);
        }
      }
    }
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = hh * 16 + nt * 8 + 2 * cq;
      red[warp][g][col] = acc[hh][nt][0];
      red[warp][g][col + 1] = acc[hh][nt][1];
      red[warp][g + 8][col] = acc[hh][nt][2];
      red[warp][g + 8][col + 1] = acc[hh][nt][3];
    }
  __syncthreads();
  for (int e = threadIdx.x; e < 16 * 32; e += 256) {
    const int row = e >> 5, j = e & 31;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += red[w][row][j];
    const int t = r0 + row;
    if (t < T) {
      if (nsplit > 1) {
        part[((size_t)split * T + t) * 32 + j] = v;
        continue;
      }
      const float sv = s * v;
      if (out_f32) out_f32[(size_t)t * 32 + j] = sv;
      if (out_ext) {
        out_ext[(size_t)t * 64 + j] = __float2bfloat16_rn(sv);
        out_ext[(size_t)t * 64 + 32 + j] = __float2bfloat16_rn(0.f);
      }
    }
  }
}

// Sum of the K-slice partials in slice order, then the scale and the outputs.
__global__ void lora_proj_reduce_kernel(const float* __restrict__ part, int nsplit, int T, float s,
                                        float* __restrict__ out_f32, __nv_bfloat16* __restrict__ out_ext) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= T * 32) return;
  const int t = e >> 5, j = e & 31;
  float v = 0.f;
  for (int k = 0; k < nsplit; ++k) v += part[(size_t)k * T * 32 + e];
  const float sv = s * v;
  if (out_f32) out_f32[e] = sv;
  if (out_ext) {
    out_ext[(size_t)t * 64 + j] = __float2bfloat16_rn(sv);
    out_ext[(size_t)t * 64 + 32 + j] = __float2bfloat16_rn(0.f);
  }
}

// Partial outer products over a slice of rows (the LoRA weight gradients dB = dY^T u
// and dA = du^T x, reduced over tokens without atomics):
//   part[chunk][c][j] = sum_{t in chunk} X[t, c] * U[t, j]     (c < ncols, j < 16)
// X bf16 [T, ldx] (16-byte aligned rows, ncols % 8 == 0); U fp32 or bf16 [T, ldu], of
// which only the first r columns are read (the sums of columns r..15 are zero).
// As a matrix product out = X^T U over the chunk's rows, on the tensor cores (mma.sync
// m16n8k16, fp32 accumulation): a block takes a 64-column strip of one chunk, in
// sub-tiles of up to 128 rows staged in shared memory (X as [t][c], read transposed by
// ldmatrix as the A operand; U transposed to [j][t] as the B operand).  A bf16 U is
// exact; an fp32 U is split into u_hi = bf16(u) and u_lo = bf16(u - u_hi), two MMAs, so
// about 16 of its mantissa bits take part (the products themselves are exact in fp32).
// Warp w takes columns 16 (w & 3) .. + 15 and j = 8 (w >> 2) .. + 7; every sum runs
// over the chunk's rows in a fixed order.
__global__ void __launch_bounds__(256) lora_outer_partial_kernel(const __nv_bfloat16* __restrict__ X, long long ldx,
                                                                 int ncols, const float* __restrict__ Uf,
                                                                 const __nv_bfloat16* __restrict__ Ub, int ldu, int r,
                                                                 int T, int rows_per_chunk, float* __restrict__ part) {
  constexpr int XS = 64 + 8, US = 128 + 8;   // padded row pitches (conflict-free ldmatrix)
  __shared__ __align__(16) __nv_bfloat16 xs[128][XS];
  __shared__ __align__(16) __nv_bfloat16 uh[16][US];
  __shared__ __align__(16) __nv_bfloat16 ul[16][US];
  const int c0 = blockIdx.x * 64;
  const int chunk = blockIdx.y;
  const int t0 = chunk * rows_per_chunk, t1 = min(T, t0 + rows_per_chunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = warp & 3, nt = warp >> 2;
  const bool split = Uf != nullptr;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int tb = t0; tb < t1; tb += 128) {
    const int nrow = min(128, t1 - tb);
    uint4 xv[4];
    float uv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = threadIdx.x + i * 256, tt = e >> 3, col = c0 + (e & 7) * 8;
      xv[i] = (tt < nrow && col < ncols) ? *reinterpret_cast<const uint4*>(X + (size_t)(tb + tt) * ldx + col)
                                         : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = threadIdx.x + i * 256, tt = e >> 4, j = e & 15;
      uv[i] = 0.f;
      if (tt < nrow && j < r) uv[i] = split ? Uf[(size_t)(tb + tt) * ldu + j] : bf2f(Ub[(size_t)(tb + tt) * ldu + j]);
    }
    __syncthreads();   // the previous sub-tile's readers are done
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = threadIdx.x + i * 256;
      *reinterpret_cast<uint4*>(&xs[e >> 3][(e & 7) * 8]) = xv[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = threadIdx.x + i * 256, tt = e >> 4, j = e & 15;
      const __nv_bfloat16 hi = __float2bfloat16_rn(uv[i]);
      uh[j][tt] = hi;
      ul[j][tt] = __float2bfloat16_rn(uv[i] - __bfloat162float(hi));
    }
    __syncthreads();
    const int ksteps = (nrow + 15) >> 4;   // rows past nrow are zero in both operands
    for (int ks = 0; ks < ksteps; ++ks) {
      const int k0 = ks * 16;
      // A = X^T (16 columns x 16 rows): four 8 x 8 blocks read transposed from [t][c]
      uint32_t a[4];
      {
        const int mm = ((lane >> 3) & 1) * 8, kk = (lane >> 4) * 8;
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                     : "r"(smem_u32(&xs[k0 + kk + (lane & 7)][mt * 16 + mm])));
      }
      // B = U (16 rows x 8 j), stored [j][t]: two 8 x 8 blocks (k 0-7, 8-15)
      uint32_t bh[2], bl[2];
      {
        const __nv_bfloat16* ph = &uh[nt * 8 + (lane & 7)][k0 + ((lane >> 3) & 1) * 8];
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                     : "=r"(bh[0]), "=r"(bh[1]) : "r"(smem_u32(ph)));
      }
      mma_16816_bf16(acc, a, bh[0], bh[1]);
      if (split) {
        const __nv_bfloat16* pl = &ul[nt * 8 + (lane & 7)][k0 + ((lane >> 3) & 1) * 8];
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                     : "=r"(bl[0]), "=r"(bl[1]) : "r"(smem_u32(pl)));
        mma_16816_bf16(acc, a, bl[0], bl[1]);
      }
    }
  }
  // accumulator (16 columns x 8 j): thread (g, q) holds columns g, g + 8 and j 2q, 2q+1
  const int g = lane >> 2, q = lane & 3;
  const int j = nt * 8 + 2 * q;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = c0 + mt * 16 + g + 8 * h;
    if (c < ncols)
      *reinterpret_cast<float2*>(part + ((size_t)chunk * ncols + c) * 16 + j) = make_float2(acc[2 * h], acc[2 * h + 1]);
  }
}

// out (+)= sum over chunks, in chunk order.  layout 0: out[c * r + j] (B-shaped [ncols, r]);
// layout 1: out[j * ncols + c] (A-shaped [r, ncols]).
__global__ void lora_outer_reduce_kernel(const float* __restrict__ part, int nchunks, int ncols, int r,
                                         int layout, int accumulate, float* __restrict__ out) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= ncols * r) return;
  const int c = layout == 0 ? e / r : e % ncols;
  const int j = layout == 0 ? e % r : e / ncols;
  float s = 0.f;
  for (int k = 0; k < nchunks; ++k) s += part[((size_t)k * ncols + c) * 16 + j];
  out[e] = accumulate ? out[e] + s : s;
}

// B_ext [N, 64] for the forward extra stage: rows of B_q in columns 0..r-1 for the
// q rows, rows of B_v in columns 16..16+r-1 for the v rows, zero elsewhere.
__global__ void build_ext_fwd_kernel(const __nv_bfloat16* __restrict__ bq, int q0, int nq,
                                     const __nv_bfloat16* __restrict__ bv, int v0, int nv, int r, int N,
                                     __nv_bfloat16* __restrict__ ext) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= N * 64) return;
  const int n = e >> 6, c = e & 63;
  float v = 0.f;
  if (bq && c < 16 && c < r && n >= q0 && n < q0 + nq) v = bf2f(bq[(size_t)(n - q0) * r + c]);
  if (bv && c >= 16 && c < 16 + r && n >= v0 && n < v0 + nv) v = bf2f(bv[(size_t)(n - v0) * r + (c - 16)]);
  ext[e] = __float2bfloat16_rn(v);
}

// A_ext [K, 64] for the backward extra stage: row k = [A_q[:, k] | A_v[:, k] | 0].
__global__ void build_ext_bwd_kernel(const __nv_bfloat16* __restrict__ aq, const __nv_bfloat16* __restrict__ av,
                                     int r, int K, __nv_bfloat16* __restrict__ ext) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= K * 64) return;
  const int k = e >> 6, c = e & 63;
  float v = 0.f;
  if (aq && c < r) v = bf2f(aq[(size_t)c * K + k]);
  if (av && c >= 16 && c < 16 + r) v = bf2f(av[(size_t)(c - 16) * K + k]);
  ext[e] = __float2bfloat16_rn(v);
}

__global__ void cast_f32_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    out[i] = __float2bfloat16_rn(in[i]);
}

}  // namespace ls
