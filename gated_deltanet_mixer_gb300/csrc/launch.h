// launch.h -- internal interface between the C ABI (api.cu) and the kernels.
// Arguments arrive here already validated (sizes, alignment, aliasing).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kDHead = 128;  // Dk = Dv accepted by the kernels

struct Dims {
  int B, T, Hk, Hv;     // Dk = Dv = 128
  long long C;          // 2*Hk*128 + Hv*128
  float eps_l2, eps_norm, q_scale;
};

struct PrefillArgs {
  Dims d;
  const void *qkv_pre, *z;
  const float *g, *beta;
  const void *conv_w, *norm_w;
  const float *S0;      // may be null (zeros)
  const void *conv0;    // may be null (zeros)
  void *o;
  float *S_T;
  void *conv_T;
  unsigned int *err;    // device error word
};

struct DecodeArgs {
  Dims d;               // d.T == 1
  const void *qkv_pre, *z;
  const float *g, *beta;
  const void *conv_w, *norm_w;
  float *S;
  const void *conv_in;
  void *conv_out;
  void *o;
  unsigned int *err;
};

// Each returns the cudaGetLastError() of its launch.
cudaError_t launch_decode(const DecodeArgs &a, bool bf16, cudaStream_t s);
cudaError_t launch_prefill(const PrefillArgs &a, bool bf16, cudaStream_t s);          // token-serial
cudaError_t launch_prefill_chunked(const PrefillArgs &a, bool bf16, cudaStream_t s);  // chunked WY, tcgen05

// Device error bits (the error word is OR-ed).
constexpr unsigned int kErrTimeout = 1u;

}  // namespace gdn
