// gdn_device.cuh -- device helpers shared by the libgdn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kD = 128;  // Dk = Dv: the only head width the kernels take

// ---- io element access (io tensors are fp32 or bf16; math is fp32) --------
__device__ __forceinline__ float ld_io(const float *p) { return *p; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_io(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_io(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// Four consecutive io elements (8- or 16-byte aligned by construction).
__device__ __forceinline__ float4 ld_io4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld_io4(const __nv_bfloat16 *p) {
  uint2 u = *reinterpret_cast<const uint2 *>(p);
  float4 f;
  f.x = __uint_as_float(u.x << 16);
  f.y = __uint_as_float(u.x & 0xffff0000u);
  f.z = __uint_as_float(u.y << 16);
  f.w = __uint_as_float(u.y & 0xffff0000u);
  return f;
}
__device__ __forceinline__ void st_io4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void st_io4(__nv_bfloat16 *p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = u;
}

// The write gate and log decay of element i (head h) of a [token][Hv] gate
// tensor: given, or from the raw projections ("How Qwen3.5 works" section
// 9.5: beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias), in fp32).
// neg_exp_A = -exp(A_log[h]).
__device__ __forceinline__ void raw_gate_math(float a, float b, float neg_exp_A, float dt_bias, float &g,
                                              float &beta) {
  const float x = a + dt_bias;
  const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));  // softplus without overflow
  g = neg_exp_A * sp;
  beta = 1.0f / (1.0f + expf(-b));
}
template <typename IO, typename Src>
__device__ __forceinline__ void gate_at(const Src &s, long long i, int h, float &g, float &beta) {
  if (s.g) {
    g = s.g[i];
    beta = s.beta[i];
  } else {
    raw_gate_math(ld_io(static_cast<const IO *>(s.a) + i), ld_io(static_cast<const IO *>(s.b) + i),
                  -expf(s.A_log[h]), s.dt_bias[h], g, beta);
  }
}

// Longest-first placement of packed sequences (cu_seqlens[0..B]): returns
// the sequence of rank `slot` when the sequences are ordered by length,
// longest first, ties by index.  CTAs are dispatched in index order, so CTA
// slots taking sequences in this order start the longest work first.  The
// order is a permutation even for malformed offsets (their rows are then
// rejected by the caller).  All threads of the block must call it; `scratch`
// is shared memory for B + 2 ints; B <= kLongestFirstMax.
constexpr int kLongestFirstMax = 512;
__device__ __forceinline__ int longest_first(const int *cu, int B, int slot, int *scratch) {
  int *len = scratch, *pick = scratch + B;
  for (int s = threadIdx.x; s < B; s += blockDim.x) len[s] = cu[s + 1] - cu[s];
  if (threadIdx.x == 0) *pick = slot;  // replaced below; keeps the result defined
  __syncthreads();
  for (int s = threadIdx.x; s < B; s += blockDim.x) {
    const int ls = len[s];
    int rank = 0;
    for (int j = 0; j < B; ++j) {
      const int lj = len[j];
      rank += (lj > ls) || (lj == ls && j < s);
    }
    if (rank == slot) *pick = s;
  }
  __syncthreads();
  const int res = *pick;
  __syncthreads();
  return res;
}

// silu(x) = x * sigmoid(x)
__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// One halving stage of the transposed warp reduction below.
template <int HALF>
__device__ __forceinline__ void tr_stage(float (&a)[32], int lane) {
  const bool upper = (lane & HALF) != 0;
#pragma unroll
  for (int i = 0; i < HALF; ++i) {
    float send = upper ? a[i] : a[i + HALF];
    float keep = upper ? a[i + HALF] : a[i];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, HALF);
  }
}

// 32 partial sums per lane -> lane L returns the warp-wide total of a[L].
// 31 shuffles instead of 160 for 32 separate butterfly reductions.
__device__ __forceinline__ float transpose_reduce32(float (&a)[32], int lane) {
  tr_stage<16>(a, lane);
  tr_stage<8>(a, lane);
  tr_stage<4>(a, lane);
  tr_stage<2>(a, lane);
  tr_stage<1>(a, lane);
  return a[0];
}

// Streaming (evict-first) 16-byte global access for state rows touched once.
__device__ __forceinline__ float4 ld_stream(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ void st_stream(float *p, float4 v) { __stcs(reinterpret_cast<float4 *>(p), v); }

}  // namespace gdn
