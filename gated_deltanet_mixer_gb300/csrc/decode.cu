// decode.cu -- one decode token for B sequences: the memory-bound step.
//
// One CTA per (sequence b, value head h), 8 warps.  The 128 x 128 fp32 state
// of the pair is streamed through registers exactly once: each warp owns 16
// state rows (row = value index i, key index j contiguous), loads them as
// float4 per lane, forms both S k^ and S q^ in the same pass, and writes the
// updated rows straight back.  Row i of the update only needs v[i], so no
// block-wide barrier sits between loading and storing the state.
//
// Per token ("How Qwen3.5 works" section 9.6, decay -> predict -> correct ->
// read; node gdn.core of the Qwen3.8-27B spec for the v x k orientation):
//   alpha = e^g,  p = alpha S k^,  delta = beta (v - p),
//   S' = alpha S + delta k^^T,  o = S' q^ = alpha S q^ + delta (k^ . q^)
// followed by the per-head gated RMSNorm (node gdn.norm).
#include "gdn_device.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 16;

// silu(conv) of channel c for the new token; also shifts the window of c
// into conv_out when `write_window` is set.
template <typename IO>
__device__ __forceinline__ float conv_token(const IO *win, const IO *x, const IO *conv_w, IO *wout,
                                            long long C, long long c, bool write_window) {
  float x0 = ld_io(win + c), x1 = ld_io(win + C + c), x2 = ld_io(win + 2 * C + c);
  float x3 = ld_io(x + c);
  float4 w = ld_io4(conv_w + 4 * c);
  float acc = w.x * x0;
  acc = fmaf(w.y, x1, acc);
  acc = fmaf(w.z, x2, acc);
  acc = fmaf(w.w, x3, acc);
  if (write_window) {
    // raw values are copied bit-exactly (same io type)
    wout[c] = win[C + c];
    wout[C + c] = win[2 * C + c];
    wout[2 * C + c] = x[c];
  }
  return silu(acc);
}

template <typename IO, bool kRawGates>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(DecodeArgs a) {
  const Dims d = a.d;
  const int unit = blockIdx.x;
  const int b = unit / d.Hv, h = unit % d.Hv;
  const int r = d.Hv / d.Hk, kh = h / r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long C = d.C;

  __shared__ __align__(16) float s_q[kD];
  __shared__ __align__(16) float s_k[kD];
  __shared__ float s_v[kD];
  __shared__ float s_o[kD];
  __shared__ float s_red[8][2];
  __shared__ float s_kq;

  const IO *x = static_cast<const IO *>(a.qkv_pre) + (long long)b * C;
  const IO *win = static_cast<const IO *>(a.conv_in) + (long long)b * 3 * C;
  IO *wout = static_cast<IO *>(a.conv_out) + (long long)b * 3 * C;
  const IO *cw = static_cast<const IO *>(a.conv_w);

  // ---- front end: conv + SiLU (q, k of key head kh; v of head h), L2 norms
  float qraw = 0.f, kraw = 0.f;
  if (tid < kD) {
    const bool owner = (h % r) == 0;  // one CTA per key head shifts its q/k window
    qraw = conv_token(win, x, cw, wout, C, (long long)kh * kD + tid, owner);
    kraw = conv_token(win, x, cw, wout, C, (long long)d.Hk * kD + (long long)kh * kD + tid, owner);
  } else {
    const int i = tid - kD;
    s_v[i] = conv_token(win, x, cw, wout, C, 2LL * d.Hk * kD + (long long)h * kD + i, true);
  }
  float sq = warp_sum(qraw * qraw), sk = warp_sum(kraw * kraw);
  if (lane == 0) {
    s_red[warp][0] = sq;
    s_red[warp][1] = sk;
  }
  __syncthreads();
  if (tid < kD) {
    float tq = s_red[0][0] + s_red[1][0] + s_red[2][0] + s_red[3][0];
    float tk = s_red[0][1] + s_red[1][1] + s_red[2][1] + s_red[3][1];
    s_q[tid] = qraw * rsqrtf(tq + d.eps_l2) * d.q_scale;
    s_k[tid] = kraw * rsqrtf(tk + d.eps_l2);
  }
  __syncthreads();
  if (warp == 0) {
    float4 q4 = reinterpret_cast<const float4 *>(s_q)[lane];
    float4 k4 = reinterpret_cast<const float4 *>(s_k)[lane];
    float kq = warp_sum(dot4(q4, k4));
    if (lane == 0) s_kq = kq;
  }
  __syncthreads();

  // ---- state pass: each warp streams its 16 rows once
  const long long gi = (long long)b * d.Hv + h;
  float gt, beta;
  if (kRawGates) {
    gate_at<IO>(a.gate, gi, h, gt, beta);
  } else {
    gt = a.gate.g[gi];
    beta = a.gate.beta[gi];
  }
  const float alpha = expf(gt);
  const float kq = s_kq;
  const float4 k4 = reinterpret_cast<const float4 *>(s_k)[lane];
  const float4 q4 = reinterpret_cast<const float4 *>(s_q)[lane];
  float *S = a.S + gi * (kD * kD);
  const int row0 = warp * kRowsPerWarp;

  float4 s[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) s[i] = ld_stream(S + (row0 + i) * kD + 4 * lane);

  float part[32];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    part[i] = dot4(s[i], k4);
    part[16 + i] = dot4(s[i], q4);
  }
  // lane L < 16: (S k^)[row0 + L];  lane L >= 16: (S q^)[row0 + L - 16]
  const float red = transpose_reduce32(part, lane);
  const int myrow = lane & 15;
  const float Sk = __shfl_sync(0xffffffffu, red, myrow);
  const float Sq = __shfl_sync(0xffffffffu, red, myrow + 16);
  const float delta = beta * (s_v[row0 + myrow] - alpha * Sk);
  if (lane < 16) s_o[row0 + myrow] = fmaf(alpha, Sq, delta * kq);

#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const float di = __shfl_sync(0xffffffffu, delta, i);
    float4 n;
    n.x = fmaf(alpha, s[i].x, di * k4.x);
    n.y = fmaf(alpha, s[i].y, di * k4.y);
    n.z = fmaf(alpha, s[i].z, di * k4.z);
    n.w = fmaf(alpha, s[i].w, di * k4.w);
    st_stream(S + (row0 + i) * kD + 4 * lane, n);
  }
  __syncthreads();

  // ---- gated RMSNorm over the head's 128 outputs
  float ov = 0.f;
  if (tid < kD) ov = s_o[tid];
  float ss = warp_sum(ov * ov);
  if (lane == 0) s_red[warp][0] = ss;
  __syncthreads();
  if (tid < kD) {
    float tot = s_red[0][0] + s_red[1][0] + s_red[2][0] + s_red[3][0];
    float rstd = rsqrtf(tot * (1.0f / kD) + d.eps_norm);
    const long long oi = gi * kD + tid;  // [B][Hv*Dv]
    float zv = ld_io(static_cast<const IO *>(a.z) + oi);
    float wv = ld_io(static_cast<const IO *>(a.norm_w) + tid);
    st_io(static_cast<IO *>(a.o) + oi, wv * (ov * rstd) * silu(zv));
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, bool bf16, cudaStream_t s) {
  dim3 grid((unsigned)(a.d.B * a.d.Hv)), block(kThreads);
  const bool raw = a.gate.g == nullptr;
  if (bf16)
    (raw ? decode_kernel<__nv_bfloat16, true> : decode_kernel<__nv_bfloat16, false>)<<<grid, block, 0, s>>>(a);
  else
    (raw ? decode_kernel<float, true> : decode_kernel<float, false>)<<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
