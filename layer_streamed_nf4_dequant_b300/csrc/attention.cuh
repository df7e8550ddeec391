// Causal grouped-query attention: the pieces the tensor-core kernels (attention_tc.cuh)
// share, for the decoder layers of the streamed stack (the Llama/Qwen-shaped models the
// Soup pages fine-tune: Soup: Fine-Tune an 8B Model on a 4 GB GPU, "The Core Idea: Layer
// Streaming"): the sequence ranges of a packed batch, the backward's row dot products
// D = rowsum(dO o O), and the fixed-order sum of per-query-head dK / dV partials.
#pragma once
#include "common.cuh"

namespace ls {

// ------------------------------------------------------------------ sequences
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
