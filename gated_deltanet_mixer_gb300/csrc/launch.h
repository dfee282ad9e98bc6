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

// Where a token's gates come from: g and beta given, or (g == nullptr) the
// raw projections a, b (io dtype, same [token][Hv] layout) with the per-head
// parameters A_log, dt_bias [Hv].
struct GateSrc {
  const float *g, *beta;
  const void *a, *b;
  const float *A_log, *dt_bias;
};

// Fixed length: sequence b owns tokens b*T .. b*T + T - 1 of the token-major
// tensors.  Packed (cu_seqlens != nullptr): sequence b owns tokens
// cu_seqlens[b] .. cu_seqlens[b+1] - 1 and d.T is the total token count.
struct PrefillArgs {
  Dims d;
  const void *qkv_pre, *z;
  GateSrc gate;
  const void *conv_w, *norm_w;
  const float *S0;      // may be null (zeros)
  const void *conv0;    // may be null (zeros)
  void *o;
  float *S_T;
  void *conv_T;
  const int *cu_seqlens;  // may be null (fixed length)
  float *S_snap;          // may be null: the state after every token, [token][Hv][128][128]
  void *qk_ws;            // may be null: staged q^ / k^, fp16 [3][token rows][Hk][128]
                          // (q^, k^ hi, k^ lo), written by launch_prefill_qk
  unsigned int *err;      // device error word
};

// T = d.T new tokens per sequence from the cache (1 <= T <= kDecodeMaxT):
// qkv_pre [B][T][C], z and o [B][T][Hv*128], gates [B][T][Hv].
constexpr int kDecodeMaxT = 16;
struct DecodeArgs {
  Dims d;
  const void *qkv_pre, *z;
  GateSrc gate;
  const void *conv_w, *norm_w;
  float *S;             // in place
  float *S_snap;        // may be null: the state after every token, [B][T][Hv][128][128]
  const void *conv_in;
  void *conv_out;
  void *o;
  unsigned int *err;
};

// y[t, n] = sum_k x[t, k] w[n, k] (bf16 x [M][ldx], w [N][ldw]); columns
// [col_begin, col_end) of y go to out[o].ptr[row * ld + col - col_begin].
struct GemmOut {
  int col_begin, col_end;
  void *ptr;
  long long ld;
  int vec_ok;  // 16-byte stores allowed (ptr, ld and col_begin aligned)
};
constexpr int kGemmMaxOut = 4;
struct GemmArgs {
  int M, N, K;
  const void *x, *w;
  long long ldx, ldw;
  int n_out;
  GemmOut out[kGemmMaxOut];
  unsigned int *err;
};

// Each returns the cudaGetLastError() of its launch.
cudaError_t launch_decode(const DecodeArgs &a, bool bf16, cudaStream_t s);
cudaError_t launch_prefill(const PrefillArgs &a, bool bf16, cudaStream_t s);          // token-serial
cudaError_t launch_prefill_chunked(const PrefillArgs &a, bool bf16, cudaStream_t s);  // chunked WY, tcgen05
// q^ / k^ into a.qk_ws (bf16 io); also zeroes nzero ints at `zero` (may be null).
cudaError_t launch_prefill_qk(const PrefillArgs &a, cudaStream_t s, int *zero = nullptr, long long nzero = 0);

// The chunk-parallel / sequential prefill (prefill_split.cu).  Chunk slots
// index the workspace: fixed length, slot = b * nch + n; packed sequences,
// slot = (cu[b] >> 6) + b + n.  A work item is (slot, value head), item =
// slot * Hv + h, and owns kSplitItemBytes of workspace across four arrays:
//   ws_u   [items][128 v][64 j]  fp32   U^T
//   ws_nw  [items][128 k][64 j]  fp16   -W^T
//   ws_m   [items][64 i][64 j]   fp16   M = (Q K^T) o R (lower, diagonal included)
//   ws_vec [items][2][64]        fp32   d_i = e^{G_i}, Gamma_j = e^{G_last - G_j}
//   flags  [items]               int32  0, then 1 once the item's outputs are written
//                                       (zeroed by launch_prefill_qk; read when both
//                                       parts run in one launch)
// The staged q^ / k^ (qk_ws, from launch_prefill_qk) must be in place first.
struct SplitArgs {
  int B, T;        // sequences; tokens per sequence (fixed length) or in total (packed)
  int nch, nslots; // chunks per sequence (fixed length); chunk slots
  const int *cu;   // cu_seqlens or null
  float *ws_u;
  void *ws_nw, *ws_m;
  float *ws_vec;
  int *flags;
};
constexpr size_t kSplitItemBytes = 32768 + 16384 + 8192 + 512 + 4;
// Work items of a call (tokens: B*T fixed length, T packed); sets nslots, nch.
long long split_items(const Dims &d, long long tokens, bool packed, int *nslots, int *nch);
cudaError_t launch_prefill_split(const PrefillArgs &a, const SplitArgs &s, cudaStream_t st);

// The library's device scratch (GDN_STATIC_SCRATCH_BYTES) on the current
// device; its address is looked up once per device.
cudaError_t static_scratch(void **ptr);
cudaError_t launch_gemm(const GemmArgs &a, int num_sms, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned int *err, unsigned long long limit_ns, cudaStream_t s);

// Device error bits (the error word is OR-ed).
constexpr unsigned int kErrTimeout = 1u;  // a bounded wait gave up
constexpr unsigned int kErrSeqlens = 2u;  // packed-sequence offsets out of order or range
constexpr unsigned int kErrBounds = 4u;   // a GDN_CHECKS bounds check failed

// GDN_CHECKS builds check every thread-issued global store of the prefill
// (q/k, prep and sequential kernels) and decode kernels against its buffer:
// `end` is one past the last element the store writes, `size` the buffer's
// element count.  A failed check sets kErrBounds in the error word and the
// caller skips the store; there is no trap.  Other builds compile it away.
__device__ __forceinline__ bool in_bounds(long long end, long long size, unsigned int *err) {
#ifdef GDN_CHECKS
  if (end > size || end <= 0) {
    atomicOr(err, kErrBounds);
    return false;
  }
#else
  (void)end;
  (void)size;
  (void)err;
#endif
  return true;
}

}  // namespace gdn
