// prefill_recurrent.cu -- token-serial prefill: the recurrence of node gdn.core
// (Qwen3.8-27B spec) run token by token with the state held in registers.
//
// One CTA per (sequence b, value head h), 8 warps; warp w owns state rows
// 16w .. 16w+15 for the whole sequence (float4 per lane per row), so the
// recurrence needs no block barrier.  Tokens are processed in blocks of 32:
//   1. conv + SiLU: each thread slides the 4-wide window of the channels it
//      owns (q and k of key head h/r, or v of head h) through the block,
//   2. L2 norms of q and k per token (one warp per token),
//   3. the serial gated delta rule over the block's tokens,
//   4. the per-head gated RMSNorm of the block's outputs (node gdn.norm).
// It also serves packed variable-length batches, raw gate projections and
// per-token state snapshots (each warp stores its rows after every token),
// and T-token decoding from the cache (S0 == S_T).
#include "gdn_device.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = 16;
constexpr int kTB = 32;  // tokens per block
constexpr size_t kSmemBytes = (4 * kTB * kD + 3 * kTB) * sizeof(float);

struct Window {
  float x0, x1, x2;  // raw inputs of the three previous tokens, oldest first
};

template <typename IO>
__device__ __forceinline__ Window load_window(const IO *conv0, long long C, long long c) {
  Window w{0.f, 0.f, 0.f};
  if (conv0) {
    w.x0 = ld_io(conv0 + c);
    w.x1 = ld_io(conv0 + C + c);
    w.x2 = ld_io(conv0 + 2 * C + c);
  }
  return w;
}

__device__ __forceinline__ float conv_step(Window &w, float4 taps, float x) {
  float acc = taps.x * w.x0;
  acc = fmaf(taps.y, w.x1, acc);
  acc = fmaf(taps.z, w.x2, acc);
  acc = fmaf(taps.w, x, acc);
  w.x0 = w.x1;
  w.x1 = w.x2;
  w.x2 = x;
  return silu(acc);
}

template <typename IO>
__device__ __forceinline__ void store_window(IO *conv_T, long long C, long long c, const Window &w) {
  st_io(conv_T + c, w.x0);
  st_io(conv_T + C + c, w.x1);
  st_io(conv_T + 2 * C + c, w.x2);
}

template <typename IO>
__global__ void __launch_bounds__(kThreads, 1) prefill_recurrent_kernel(PrefillArgs a) {
  const Dims d = a.d;
  const int unit = blockIdx.x;
  const int h = unit % d.Hv;
  int b = unit / d.Hv;
  const int r = d.Hv / d.Hk, kh = h / r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long C = d.C;
  extern __shared__ __align__(16) float smem[];
  if (a.cu_seqlens && d.B <= kLongestFirstMax)  // packed: the longest sequences first
    b = longest_first(a.cu_seqlens, d.B, b, reinterpret_cast<int *>(smem));
  // This sequence's tokens: rows bos .. bos + T - 1 of the token-major tensors.
  long long bos;
  int T;
  if (a.cu_seqlens) {
    const int lo = a.cu_seqlens[b], hi = a.cu_seqlens[b + 1];
    if (lo < 0 || hi < lo || hi > d.T) {  // unusable offsets: leave this sequence untouched
      if (tid == 0) atomicOr(a.err, kErrSeqlens);
      return;
    }
    bos = lo;
    T = hi - lo;
  } else {
    bos = (long long)b * d.T;
    T = d.T;
  }

  float *s_q = smem;              // [kTB][128] normalised, scaled query
  float *s_k = s_q + kTB * kD;    // [kTB][128] normalised key
  float *s_v = s_k + kTB * kD;    // [kTB][128] value
  float *s_o = s_v + kTB * kD;    // [kTB][128] core output
  float *s_alpha = s_o + kTB * kD;
  float *s_beta = s_alpha + kTB;
  float *s_kq = s_beta + kTB;

  const IO *x = static_cast<const IO *>(a.qkv_pre) + bos * C;
  const IO *cw = static_cast<const IO *>(a.conv_w);
  const IO *conv0 = a.conv0 ? static_cast<const IO *>(a.conv0) + (long long)b * 3 * C : nullptr;

  // Channel ownership for the front end.
  const bool qk_thread = tid < kD;
  const long long cq = (long long)kh * kD + tid;
  const long long ck = (long long)d.Hk * kD + (long long)kh * kD + tid;
  const long long cv = 2LL * d.Hk * kD + (long long)h * kD + (tid - kD);
  Window wq{}, wk{}, wv{};
  float4 tq{}, tk{}, tv{};
  if (qk_thread) {
    wq = load_window(conv0, C, cq);
    wk = load_window(conv0, C, ck);
    tq = ld_io4(cw + 4 * cq);
    tk = ld_io4(cw + 4 * ck);
  } else {
    wv = load_window(conv0, C, cv);
    tv = ld_io4(cw + 4 * cv);
  }

  // State rows in registers.
  const long long gi0 = (long long)b * d.Hv + h;
  const int row0 = warp * kRowsPerWarp;
  float4 s[kRowsPerWarp];
  if (a.S0) {
    const float *S0 = a.S0 + gi0 * (kD * kD);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) s[i] = ld_stream(S0 + (row0 + i) * kD + 4 * lane);
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  for (int t0 = 0; t0 < T; t0 += kTB) {
    const int nt = min(kTB, T - t0);
    // 1. conv + SiLU
    for (int tt = 0; tt < nt; ++tt) {
      const IO *xt = x + (long long)(t0 + tt) * C;
      if (qk_thread) {
        s_q[tt * kD + tid] = conv_step(wq, tq, ld_io(xt + cq));
        s_k[tt * kD + tid] = conv_step(wk, tk, ld_io(xt + ck));
      } else {
        s_v[tt * kD + (tid - kD)] = conv_step(wv, tv, ld_io(xt + cv));
      }
    }
    if (tid < nt) {
      float gt, bt;
      gate_at<IO>(a.gate, (bos + t0 + tid) * d.Hv + h, h, gt, bt);
      s_alpha[tid] = expf(gt);
      s_beta[tid] = bt;
    }
    __syncthreads();
    // 2. L2 norms
    for (int tt = warp; tt < nt; tt += kWarps) {
      float4 q4 = reinterpret_cast<float4 *>(s_q + tt * kD)[lane];
      float4 k4 = reinterpret_cast<float4 *>(s_k + tt * kD)[lane];
      const float fq = rsqrtf(warp_sum(dot4(q4, q4)) + d.eps_l2) * d.q_scale;
      const float fk = rsqrtf(warp_sum(dot4(k4, k4)) + d.eps_l2);
      q4.x *= fq; q4.y *= fq; q4.z *= fq; q4.w *= fq;
      k4.x *= fk; k4.y *= fk; k4.z *= fk; k4.w *= fk;
      reinterpret_cast<float4 *>(s_q + tt * kD)[lane] = q4;
      reinterpret_cast<float4 *>(s_k + tt * kD)[lane] = k4;
      const float kq = warp_sum(dot4(q4, k4));
      if (lane == 0) s_kq[tt] = kq;
    }
    __syncthreads();
    // 3. the recurrence, token by token; each warp on its own rows
    for (int tt = 0; tt < nt; ++tt) {
      const float4 k4 = reinterpret_cast<const float4 *>(s_k + tt * kD)[lane];
      const float4 q4 = reinterpret_cast<const float4 *>(s_q + tt * kD)[lane];
      const float alpha = s_alpha[tt], beta = s_beta[tt], kq = s_kq[tt];
      float part[32];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        part[i] = dot4(s[i], k4);
        part[16 + i] = dot4(s[i], q4);
      }
      const float red = transpose_reduce32(part, lane);
      const int myrow = lane & 15;
      const float Sk = __shfl_sync(0xffffffffu, red, myrow);
      const float Sq = __shfl_sync(0xffffffffu, red, myrow + 16);
      const float delta = beta * (s_v[tt * kD + row0 + myrow] - alpha * Sk);
      if (lane < 16) s_o[tt * kD + row0 + myrow] = fmaf(alpha, Sq, delta * kq);
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const float di = __shfl_sync(0xffffffffu, delta, i);
        s[i].x = fmaf(alpha, s[i].x, di * k4.x);
        s[i].y = fmaf(alpha, s[i].y, di * k4.y);
        s[i].z = fmaf(alpha, s[i].z, di * k4.z);
        s[i].w = fmaf(alpha, s[i].w, di * k4.w);
      }
      if (a.S_snap) {
        float *snap = a.S_snap + ((bos + t0 + tt) * d.Hv + h) * (kD * kD);
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) st_stream(snap + (row0 + i) * kD + 4 * lane, s[i]);
      }
    }
    __syncthreads();
    // 4. gated RMSNorm, one warp per token
    const float4 w4 = ld_io4(static_cast<const IO *>(a.norm_w) + 4 * lane);
    for (int tt = warp; tt < nt; tt += kWarps) {
      const float4 o4 = reinterpret_cast<const float4 *>(s_o + tt * kD)[lane];
      const float rstd = rsqrtf(warp_sum(dot4(o4, o4)) * (1.0f / kD) + d.eps_norm);
      const long long oi = ((bos + t0 + tt) * d.Hv + h) * kD + 4 * lane;
      const float4 z4 = ld_io4(static_cast<const IO *>(a.z) + oi);
      float4 y;
      y.x = w4.x * (o4.x * rstd) * silu(z4.x);
      y.y = w4.y * (o4.y * rstd) * silu(z4.y);
      y.z = w4.z * (o4.z * rstd) * silu(z4.z);
      y.w = w4.w * (o4.w * rstd) * silu(z4.w);
      st_io4(static_cast<IO *>(a.o) + oi, y);
    }
    // s_o is rewritten only after the next block's two barriers.
  }

  float *ST = a.S_T + gi0 * (kD * kD);
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) st_stream(ST + (row0 + i) * kD + 4 * lane, s[i]);

  IO *cT = static_cast<IO *>(a.conv_T) + (long long)b * 3 * C;
  if (qk_thread) {
    if ((h % r) == 0) {
      store_window(cT, C, cq, wq);
      store_window(cT, C, ck, wk);
    }
  } else {
    store_window(cT, C, cv, wv);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, bool bf16, cudaStream_t s) {
  dim3 grid((unsigned)(a.d.B * a.d.Hv)), block(kThreads);
  cudaError_t e;
  if (bf16) {
    e = cudaFuncSetAttribute(prefill_recurrent_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_recurrent_kernel<__nv_bfloat16><<<grid, block, kSmemBytes, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(prefill_recurrent_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_recurrent_kernel<float><<<grid, block, kSmemBytes, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
