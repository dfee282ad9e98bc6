// decode.cu -- new tokens for B sequences from the cache: the memory-bound
// step.  decode1_kernel takes one token (the common case, no snapshots);
// decode_kernel takes T <= kDecodeMaxT tokens and can keep the state after
// every token.
//
// 8 warps per CTA.  The 128 x 128 fp32 state of a (sequence b, value head h)
// pair is streamed through registers exactly once: each warp owns 16 state
// rows (row = value index i, key index j contiguous), per token forms both
// S k^ and S q^ in the same pass and updates the rows in registers; the
// final rows (and, when asked, the rows after every token) are written
// straight back.  Row i of the update only needs v[i], so no block-wide
// barrier sits inside the state pass.  decode1_kernel: one CTA per pair,
// lane L holding columns 4L .. 4L + 3 of the warp's rows.  decode_kernel:
// persistent (two CTAs per SM walking the pairs), the next pair's state
// (and, with bf16 io, its raw rows, window, conv weights and z) copied into
// shared memory while the current pair's T serial token steps run, and lane
// (rg, cg) holding 4 rows x 16 columns, so that a token's dot products reduce
// over 8 lanes.
//
// Per token ("How Qwen3.5 works" section 9.6, decay -> predict -> correct ->
// read; node gdn.core of the Qwen3.8-27B spec for the v x k orientation):
//   alpha = e^g,  p = alpha S k^,  delta = beta (v - p),
//   S' = alpha S + delta k^^T,  o = S' q^ = alpha S q^ + delta (k^ . q^)
// followed by the per-head gated RMSNorm (node gdn.norm).
#include <cstddef>

#include "gdn_device.cuh"
#include "launch.h"
#include "tma_host.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = 16;

// silu(conv) of channel c for the new token; also shifts the window of c
// into conv_out when `write_window` is set.
template <typename IO>
__device__ __forceinline__ float conv_token(const IO *win, const IO *x, const IO *conv_w, IO *wout,
                                            long long C, long long c, bool write_window, long long wout_end,
                                            long long win_size, unsigned int *err) {
  float x0 = ld_io(win + c), x1 = ld_io(win + C + c), x2 = ld_io(win + 2 * C + c);
  float x3 = ld_io(x + c);
  float4 w = ld_io4(conv_w + 4 * c);
  float acc = w.x * x0;
  acc = fmaf(w.y, x1, acc);
  acc = fmaf(w.z, x2, acc);
  acc = fmaf(w.w, x3, acc);
  if (write_window && in_bounds(wout_end + 2 * C + c + 1, win_size, err)) {
    // raw values are copied bit-exactly (same io type)
    wout[c] = win[C + c];
    wout[C + c] = win[2 * C + c];
    wout[2 * C + c] = x[c];
  }
  return silu(acc);
}

// alpha s + di k for one state row (fmaf(alpha, s, di * k) per element), paired.
__device__ __forceinline__ float4 decay_update(float4 s, float alpha, float di, float4 k) {
  const float2 n01 = __ffma2_rn(make_float2(alpha, alpha), make_float2(s.x, s.y),
                                __fmul2_rn(make_float2(di, di), make_float2(k.x, k.y)));
  const float2 n23 = __ffma2_rn(make_float2(alpha, alpha), make_float2(s.z, s.w),
                                __fmul2_rn(make_float2(di, di), make_float2(k.z, k.w)));
  return make_float4(n01.x, n01.y, n23.x, n23.y);
}

template <typename IO, bool kRawGates>
__global__ void __launch_bounds__(kThreads, 2) decode1_kernel(DecodeArgs a) {
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
  const long long wbase = (long long)b * 3 * C, wsize = (long long)d.B * 3 * C;  // window offset, elements
  const long long S_size = (long long)d.B * d.Hv * kD * kD;

  // This warp's 16 state rows and this thread's z element, requested first:
  // their latency overlaps the front end's.  (Requesting the gates here too
  // measured slower.)
  const long long gi = (long long)b * d.Hv + h;
  float *S = a.S + gi * (kD * kD);
  const int row0 = warp * kRowsPerWarp;
  float4 s[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) s[i] = ld_stream(S + (row0 + i) * kD + 4 * lane);
  const float zv = tid < kD ? ld_io(static_cast<const IO *>(a.z) + gi * kD + tid) : 0.f;

  // ---- front end: conv + SiLU (q, k of key head kh; v of head h), L2 norms
  float qraw = 0.f, kraw = 0.f;
  if (tid < kD) {
    const bool owner = (h % r) == 0;  // one CTA per key head shifts its q/k window
    qraw = conv_token(win, x, cw, wout, C, (long long)kh * kD + tid, owner, wbase, wsize, a.err);
    kraw = conv_token(win, x, cw, wout, C, (long long)d.Hk * kD + (long long)kh * kD + tid, owner, wbase, wsize, a.err);
  } else {
    const int i = tid - kD;
    s_v[i] = conv_token(win, x, cw, wout, C, 2LL * d.Hk * kD + (long long)h * kD + i, true, wbase, wsize, a.err);
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
    if (in_bounds(gi * (kD * kD) + (row0 + i) * kD + 4 * lane + 4, S_size, a.err)) st_stream(S + (row0 + i) * kD + 4 * lane, n);
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
    float wv = ld_io(static_cast<const IO *>(a.norm_w) + tid);
    if (in_bounds(oi + 1, (long long)d.B * d.Hv * kD, a.err)) st_io(static_cast<IO *>(a.o) + oi, wv * (ov * rstd) * silu(zv));
  }
}

// The T-token kernel's shared memory: the next unit's state (filled by bulk
// copies while the current unit is computed from registers), the current
// unit's token vectors, and (bf16 io) the raw inputs of the unit whose turn
// is next, also by asynchronous copy: its new rows' and window's q, k, v
// channel blocks (one TMA box each), their conv weights and its z rows.
struct DecodeSmem {
  float S[kD * kD];  // 64 KB
  // q^, k^ and v of each token; o is written over v (each warp over its own rows)
  float q[kDecodeMaxT][kD], k[kDecodeMaxT][kD], v[kDecodeMaxT][kD];
  float kq[kDecodeMaxT], g[kDecodeMaxT], b[kDecodeMaxT];
  alignas(128) uint16_t xr[3][kDecodeMaxT][kD];  // raw rows of the q, k, v blocks (bf16 io; fp32 io keeps z here)
  alignas(128) uint16_t wr[3][3][kD];            // the carried window, same blocks
  alignas(128) uint16_t cwr[3 * kD * 4];         // conv weights of those channels
  alignas(128) uint16_t zr[kDecodeMaxT][kD];     // z rows
  uint64_t bar;     // the state copy landed
  uint64_t bar_in;  // raw rows, window and conv weights landed
  uint64_t bar_z;   // z rows landed
  int stop;
};
constexpr uint32_t kStateBytes = kD * kD * 4;
constexpr size_t kDecodeSmem = sizeof(DecodeSmem) + 128;  // + alignment slack
static_assert(offsetof(DecodeSmem, S) == 0 && offsetof(DecodeSmem, q) % 16 == 0 && offsetof(DecodeSmem, xr) % 128 == 0 &&
                  offsetof(DecodeSmem, wr) % 128 == 0 && offsetof(DecodeSmem, cwr) % 128 == 0 &&
                  offsetof(DecodeSmem, zr) % 128 == 0 && offsetof(DecodeSmem, bar) % 8 == 0,
              "layout (TMA destinations 128-byte aligned)");
static_assert(sizeof(float) * kDecodeMaxT * kD <= sizeof(uint16_t) * 3 * kDecodeMaxT * kD, "fp32 z fits the raw rows");
static_assert(2 * (kDecodeSmem + 1024) <= 233472, "two CTAs per SM");

__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   umma::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(umma::smem_u32(bar))
               : "memory");
}
// silu(x) = x / (1 + 2^(-x log2 e)) on the MUFU ex2 and rcp approximations
// (relative error about 1e-6; the inputs and outputs are bf16 here).
__device__ __forceinline__ float silu_mufu(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return x * r;
}
__device__ __forceinline__ void bulk_load_state(DecodeSmem &M, const float *src) {
  umma::bar_expect_tx(&M.bar, kStateBytes);
#pragma unroll
  for (int p = 0; p < 4; ++p) bulk_copy(M.S + p * (kD * kD / 4), src + p * (kD * kD / 4), kStateBytes / 4, &M.bar);
}

// Persistent: CTA c takes the (sequence, value head) units c, c + grid, ...
// While a unit's T token steps run on its state in registers, the bulk copy
// of the CTA's next unit's state lands in shared memory, so that the state
// stream does not stop for the serial token steps; with bf16 io the next
// unit's raw inputs arrive the same way, and its gates in registers.  Two
// CTAs per SM.
//
// The tensor maps (bf16 io): tm_x over qkv_pre as rows of C (box 128 x T),
// tm_w over the carried windows as rows of C (box 128 x 3), tm_z over z as
// rows of Hv*128 (box 128 x T).  Unused (and not encoded) for fp32 io.
template <typename IO, bool kRawGates>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap tm_x,
                                                             const __grid_constant__ CUtensorMap tm_w,
                                                             const __grid_constant__ CUtensorMap tm_z) {
  constexpr bool kPre = sizeof(IO) == 2;  // inputs by asynchronous copy (bf16 io)
  extern __shared__ uint8_t decode_smem_raw[];
  DecodeSmem &M = *reinterpret_cast<DecodeSmem *>(decode_smem_raw + ((128 - (umma::smem_u32(decode_smem_raw) & 127)) & 127));
  const Dims d = a.d;
  const int T = d.T;
  const int nunits = d.B * d.Hv;
  const int r = d.Hv / d.Hk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long C = d.C;
  const IO *cw = static_cast<const IO *>(a.conv_w);
  const int row0 = warp * kRowsPerWarp;
  // fp32 io: the z rows as fp32, in the raw rows' space
  float(*zf)[kD] = reinterpret_cast<float(*)[kD]>(&M.xr[0][0]);

  if (tid == 0) {
    umma::bar_init(&M.bar, 1);
    umma::bar_init(&M.bar_in, 1);
    umma::bar_init(&M.bar_z, 1);
    M.stop = 0;
  }
  umma::fence_smem_to_async();
  __syncthreads();

  // The first channel of each of a unit's three channel blocks (q, k of its
  // key head; v of its head).
  auto chan0 = [&](int h, int seg) -> long long {
    return seg == 0 ? (long long)(h / r) * kD : seg == 1 ? (long long)(d.Hk + h / r) * kD : (long long)(2 * d.Hk + h) * kD;
  };
  // bf16 io.  Thread 0 announces a unit's copies on their barrier before a
  // block barrier; after it the copies are issued (a warp issues its lanes'
  // copies one after another, so they are spread over warps): unit u's nine
  // (raw rows and window of each channel block by TMA, conv weights by bulk
  // copy) by the warps that have no token's L2 norm (warps min(T, 7) .. 7),
  // its z rows (one TMA box) by the last warp.
  const uint32_t in_bytes = (uint32_t)(3 * T + 9) * (kD * 2) + 3 * (kD * 8), z_bytes = (uint32_t)T * (kD * 2);
  const int cw0 = T < kWarps - 1 ? T : kWarps - 1, ncw = kWarps - cw0;  // the warps issuing the input copies
  auto request_inputs = [&](int u) {
    if (warp < cw0) return;
    const int ub = u / d.Hv, uh = u % d.Hv;
    for (int i = (warp - cw0) + ncw * lane; i < 9; i += ncw * 32) {
      const int seg = i % 3;
      if (i < 3)
        umma::tma_load_3d(umma::smem_u32(&M.xr[seg][0][0]), &tm_x, (int)chan0(uh, seg), ub * T, 0, &M.bar_in);
      else if (i < 6)
        umma::tma_load_3d(umma::smem_u32(&M.wr[seg][0][0]), &tm_w, (int)chan0(uh, seg), ub * 3, 0, &M.bar_in);
      else
        bulk_copy(&M.cwr[seg * kD * 4], cw + 4 * chan0(uh, seg), kD * 8, &M.bar_in);
    }
  };
  auto request_z = [&](int u) {
    if (warp == kWarps - 1 && lane == 0)
      umma::tma_load_3d(umma::smem_u32(&M.zr[0][0]), &tm_z, (u % d.Hv) * kD, (u / d.Hv) * T, 0, &M.bar_z);
  };
  // Threads t < T: unit u's gates of token t.
  auto gates = [&](int u, float &gt, float &bt) {
    const int ub = u / d.Hv, uh = u % d.Hv;
    const long long i = ((long long)ub * T + tid) * d.Hv + uh;
    if (kRawGates) {
      gate_at<IO>(a.gate, i, uh, gt, bt);
    } else {
      gt = a.gate.g[i];
      bt = a.gate.beta[i];
    }
  };
  // Thread 0: a bounded wait; after a timeout the CTA stops at the next
  // barrier (a second bounded wait first: no copy may land after the CTA ends).
  auto wait_or_stop = [&](uint64_t *bar, uint32_t ph) {
    if (!umma::bar_wait(bar, ph)) {
      atomicOr(a.err, kErrTimeout);
      umma::bar_wait(bar, ph);
      M.stop = 1;
    }
  };

  int unit = blockIdx.x;
  uint32_t phase = 0, ph_in = 0, ph_z = 0;
  bool pending = false, pending_in = false, pending_z = false;  // copies in flight (thread 0's view)
  float ng = 0.f, nb = 0.f;  // threads t < T: the gates of the CTA's next unit (bf16 io)
  if (unit < nunits) {
    if (tid == 0) {
      bulk_load_state(M, a.S + (long long)unit * (kD * kD));
      pending = true;
    }
    if (kPre) {
      if (tid == 0) {
        umma::bar_expect_tx(&M.bar_in, in_bytes);
        umma::bar_expect_tx(&M.bar_z, z_bytes);
      }
      __syncthreads();
      request_inputs(unit);
      request_z(unit);
      pending_in = pending_z = true;
      if (tid < T) gates(unit, ng, nb);
      if (tid == 0) {
        wait_or_stop(&M.bar_in, ph_in);
        pending_in = false;
      }
      ph_in ^= 1u;
      if (tid < T) {
        M.g[tid] = ng;
        M.b[tid] = nb;
      }
      __syncthreads();
    }
  }
  for (; unit < nunits && !M.stop; unit += gridDim.x) {
    const int b = unit / d.Hv, h = unit % d.Hv, kh = h / r;
    const int next = unit + (int)gridDim.x;
    const IO *x = static_cast<const IO *>(a.qkv_pre) + (long long)b * T * C;
    const IO *win = static_cast<const IO *>(a.conv_in) + (long long)b * 3 * C;
    IO *wout = static_cast<IO *>(a.conv_out) + (long long)b * 3 * C;

    if (!kPre) {  // the gates of every token and the z rows of the gated norm
      if (tid < T) gates(unit, M.g[tid], M.b[tid]);
      for (int e = tid; e < T * (kD / 4); e += kThreads) {  // four channels per load
        const int t = e / (kD / 4), c = 4 * (e % (kD / 4));
        reinterpret_cast<float4 *>(zf[t])[c / 4] =
            ld_io4(static_cast<const IO *>(a.z) + (((long long)b * T + t) * d.Hv + h) * kD + c);
      }
    }

    // ---- front end: conv + SiLU of the T tokens, sliding the window of the
    // channel(s) this thread owns (q and k of key head kh, or v of head h);
    // with bf16 io from the raw rows in shared memory
    {
      const bool qk = tid < kD;
      const int s0 = qk ? 0 : 2, j = tid & (kD - 1);  // the channel's block and index in the raw rows (k: block 1)
      const long long c0 = qk ? (long long)kh * kD + tid : 2LL * d.Hk * kD + (long long)h * kD + (tid - kD);
      const long long c1 = (long long)d.Hk * kD + (long long)kh * kD + tid;
      auto raw = [&](const uint16_t *p) { return __uint_as_float((uint32_t)*p << 16); };  // bf16 bits -> fp32
      float w0[3], w1[3] = {0.f, 0.f, 0.f};
      float4 t0, t1 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kPre) {
        const uint2 u0 = *reinterpret_cast<const uint2 *>(&M.cwr[4 * (s0 * kD + j)]);
        t0 = make_float4(__uint_as_float(u0.x << 16), __uint_as_float(u0.x & 0xffff0000u), __uint_as_float(u0.y << 16),
                         __uint_as_float(u0.y & 0xffff0000u));
#pragma unroll
        for (int e = 0; e < 3; ++e) w0[e] = raw(&M.wr[s0][e][j]);
        if (qk) {
          const uint2 u1 = *reinterpret_cast<const uint2 *>(&M.cwr[4 * (kD + j)]);
          t1 = make_float4(__uint_as_float(u1.x << 16), __uint_as_float(u1.x & 0xffff0000u),
                           __uint_as_float(u1.y << 16), __uint_as_float(u1.y & 0xffff0000u));
#pragma unroll
          for (int e = 0; e < 3; ++e) w1[e] = raw(&M.wr[1][e][j]);
        }
      } else {
        t0 = ld_io4(cw + 4 * c0);
#pragma unroll
        for (int e = 0; e < 3; ++e) w0[e] = ld_io(win + e * C + c0);
        if (qk) {
          t1 = ld_io4(cw + 4 * c1);
#pragma unroll
          for (int e = 0; e < 3; ++e) w1[e] = ld_io(win + e * C + c1);
        }
      }
      // Tokens in batches of 8: the batch's loads are all issued before the
      // first is used, so the T tokens cost about T / 8 load latencies.
      for (int tb = 0; tb < T; tb += 8) {
        float xa[8], xb[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const bool in = tb + u < T;
          if (kPre) {
            xa[u] = in ? raw(&M.xr[s0][tb + u][j]) : 0.f;
            xb[u] = (in && qk) ? raw(&M.xr[1][tb + u][j]) : 0.f;
          } else {
            xa[u] = in ? ld_io(x + (long long)(tb + u) * C + c0) : 0.f;
            xb[u] = (in && qk) ? ld_io(x + (long long)(tb + u) * C + c1) : 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (tb + u >= T) break;
          const int t = tb + u;
          const float x0 = xa[u];
          float acc = fmaf(t0.w, x0, fmaf(t0.z, w0[2], fmaf(t0.y, w0[1], t0.x * w0[0])));
          w0[0] = w0[1];
          w0[1] = w0[2];
          w0[2] = x0;
          if (qk) {
            M.q[t][tid] = silu_mufu(acc);
            const float x1 = xb[u];
            const float acc1 = fmaf(t1.w, x1, fmaf(t1.z, w1[2], fmaf(t1.y, w1[1], t1.x * w1[0])));
            w1[0] = w1[1];
            w1[1] = w1[2];
            w1[2] = x1;
            M.k[t][tid] = silu_mufu(acc1);
          } else {
            M.v[t][tid - kD] = silu_mufu(acc);
          }
        }
      }
      // the new window: the last three raw rows (one CTA per key head shifts q/k)
      const long long wsize = (long long)d.B * 3 * C, wbase = (long long)b * 3 * C;
      if (!qk || (h % r) == 0) {
#pragma unroll
        for (int e = 0; e < 3; ++e)
          if (in_bounds(wbase + e * C + c0 + 1, wsize, a.err)) st_io(wout + e * C + c0, w0[e]);
        if (qk) {
#pragma unroll
          for (int e = 0; e < 3; ++e)
            if (in_bounds(wbase + e * C + c1 + 1, wsize, a.err)) st_io(wout + e * C + c1, w1[e]);
        }
      }
    }
    if (kPre && tid == 0 && next < nunits) umma::bar_expect_tx(&M.bar_in, in_bytes);
    __syncthreads();
    // The raw rows are read: the next unit's may land (and its gates arrive).
    if (kPre && next < nunits) {
      request_inputs(next);
      pending_in = true;
      if (tid < T) gates(next, ng, nb);
    }
    // ---- L2 norms of q and k, and k^ . q^, one warp per token
    for (int t = warp; t < T; t += kWarps) {
      float4 q4 = reinterpret_cast<const float4 *>(M.q[t])[lane];
      float4 k4 = reinterpret_cast<const float4 *>(M.k[t])[lane];
      const float fq = rsqrtf(warp_sum(dot4(q4, q4)) + d.eps_l2) * d.q_scale;
      const float fk = rsqrtf(warp_sum(dot4(k4, k4)) + d.eps_l2);
      q4.x *= fq; q4.y *= fq; q4.z *= fq; q4.w *= fq;
      k4.x *= fk; k4.y *= fk; k4.z *= fk; k4.w *= fk;
      reinterpret_cast<float4 *>(M.q[t])[lane] = q4;
      reinterpret_cast<float4 *>(M.k[t])[lane] = k4;
      const float kq = warp_sum(dot4(q4, k4));
      if (lane == 0) M.kq[t] = kq;
    }

    // ---- the state: this unit's copy landed; into registers (each warp its
    // 16 rows), then the buffer takes the next unit's
    if (tid == 0) {
      wait_or_stop(&M.bar, phase);
      pending = false;
    }
    phase ^= 1u;
    __syncthreads();
    if (M.stop) break;
    // Lane (rg, cg) = (lane >> 3, lane & 7) of a warp holds rows row0 + 4 rg
    // + i (i < 4) at columns 4 cg + 32 m + e (m, e < 4): a token's dot
    // products then reduce over the 8 lanes of a row group only, and every
    // shared-memory read of the state or of k^, q^ is conflict-free.
    const int rg = lane >> 3, cg = lane & 7;
    const int rbase = row0 + 4 * rg;
    float4 s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int m = 0; m < 4; ++m) s[i][m] = *reinterpret_cast<const float4 *>(M.S + (rbase + i) * kD + 4 * cg + 32 * m);
    __syncthreads();
    if (tid == 0 && next < nunits) {
      bulk_load_state(M, a.S + (long long)next * (kD * kD));
      pending = true;
    }

    // ---- the token steps on the registers
    const long long gi = (long long)b * d.Hv + h;
    float *S = a.S + gi * (kD * kD);
    for (int t = 0; t < T; ++t) {
      const float alpha = expf(M.g[t]), beta = M.b[t], kq = M.kq[t];
      float4 k4[4], q4[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        k4[m] = *reinterpret_cast<const float4 *>(M.k[t] + 4 * cg + 32 * m);
        q4[m] = *reinterpret_cast<const float4 *>(M.q[t] + 4 * cg + 32 * m);
      }
      // partial (S k^) and (S q^) of the lane's 4 rows over its 16 columns
      float part[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 ak = __fmul2_rn(make_float2(s[i][0].x, s[i][0].y), make_float2(k4[0].x, k4[0].y));
        float2 aq = __fmul2_rn(make_float2(s[i][0].x, s[i][0].y), make_float2(q4[0].x, q4[0].y));
        ak = __ffma2_rn(make_float2(s[i][0].z, s[i][0].w), make_float2(k4[0].z, k4[0].w), ak);
        aq = __ffma2_rn(make_float2(s[i][0].z, s[i][0].w), make_float2(q4[0].z, q4[0].w), aq);
#pragma unroll
        for (int m = 1; m < 4; ++m) {
          ak = __ffma2_rn(make_float2(s[i][m].x, s[i][m].y), make_float2(k4[m].x, k4[m].y), ak);
          aq = __ffma2_rn(make_float2(s[i][m].x, s[i][m].y), make_float2(q4[m].x, q4[m].y), aq);
          ak = __ffma2_rn(make_float2(s[i][m].z, s[i][m].w), make_float2(k4[m].z, k4[m].w), ak);
          aq = __ffma2_rn(make_float2(s[i][m].z, s[i][m].w), make_float2(q4[m].z, q4[m].w), aq);
        }
        part[i] = ak.x + ak.y;
        part[4 + i] = aq.x + aq.y;
      }
      // Sums over the row group's 8 lanes: lane cg ends with value cg,
      // i.e. (S k^)[rbase + cg] for cg < 4 and (S q^)[rbase + cg - 4] above.
#pragma unroll
      for (int o = 4; o >= 1; o >>= 1) {
        const bool up = (cg & o) != 0;
#pragma unroll
        for (int v = 0; v < o; ++v) {
          const float keep = up ? part[v + o] : part[v], send = up ? part[v] : part[v + o];
          part[v] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      const float Sq = __shfl_down_sync(0xffffffffu, part[0], 4);  // lanes cg < 4: their row's S q^
      const float delta = beta * (M.v[t][rbase + (cg & 3)] - alpha * part[0]);
      __syncwarp();  // every lane has read its v before o takes its place (this warp's rows only)
      if (cg < 4) M.v[t][rbase + cg] = fmaf(alpha, Sq, delta * kq);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float di = __shfl_sync(0xffffffffu, delta, (lane & ~7) + i);
#pragma unroll
        for (int m = 0; m < 4; ++m) s[i][m] = decay_update(s[i][m], alpha, di, k4[m]);
      }
      if (a.S_snap) {
        const long long so = (((long long)b * T + t) * d.Hv + h) * (kD * kD);
        float *snap = a.S_snap + so;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const long long off = (long long)(rbase + i) * kD + 4 * cg + 32 * m;
            if (in_bounds(so + off + 4, (long long)d.B * T * d.Hv * kD * kD, a.err)) st_stream(snap + off, s[i][m]);
          }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const long long off = (long long)(rbase + i) * kD + 4 * cg + 32 * m;
        if (in_bounds(gi * (kD * kD) + off + 4, (long long)d.B * d.Hv * kD * kD, a.err)) st_stream(S + off, s[i][m]);
      }
    if (kPre && tid == 0) {
      wait_or_stop(&M.bar_z, ph_z);
      pending_z = false;
    }
    ph_z ^= 1u;
    __syncthreads();

    // ---- gated RMSNorm over the head's 128 outputs (o in v's place), one warp per token
    const float4 w4 = ld_io4(static_cast<const IO *>(a.norm_w) + 4 * lane);
    for (int t = warp; t < T; t += kWarps) {
      const float4 o4 = reinterpret_cast<const float4 *>(M.v[t])[lane];
      const float rstd = rsqrtf(warp_sum(dot4(o4, o4)) * (1.0f / kD) + d.eps_norm);
      const long long oi = (((long long)b * T + t) * d.Hv + h) * kD + 4 * lane;  // [B][T][Hv*Dv]
      if (!in_bounds(oi + 4, (long long)d.B * T * d.Hv * kD, a.err)) continue;
      float4 z4;
      if (kPre) {
        const uint2 u = *reinterpret_cast<const uint2 *>(&M.zr[t][4 * lane]);
        z4 = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                         __uint_as_float(u.y & 0xffff0000u));
      } else {
        z4 = reinterpret_cast<const float4 *>(zf[t])[lane];
      }
      float4 y;
      y.x = w4.x * (o4.x * rstd) * silu_mufu(z4.x);
      y.y = w4.y * (o4.y * rstd) * silu_mufu(z4.y);
      y.z = w4.z * (o4.z * rstd) * silu_mufu(z4.z);
      y.w = w4.w * (o4.w * rstd) * silu_mufu(z4.w);
      st_io4(static_cast<IO *>(a.o) + oi, y);
    }
    // The next unit: its raw inputs landed (requested a unit ago) and its
    // gates take the place of this unit's; after the barrier its z rows may
    // replace these.
    if (kPre && next < nunits) {
      if (tid == 0) {
        wait_or_stop(&M.bar_in, ph_in);
        pending_in = false;
      }
      ph_in ^= 1u;
      if (tid < T) {
        M.g[tid] = ng;
        M.b[tid] = nb;
      }
      if (tid == 0) umma::bar_expect_tx(&M.bar_z, z_bytes);
    }
    __syncthreads();  // the token vectors and z rows are reused by the next unit
    if (kPre && next < nunits) {
      request_z(next);
      pending_z = true;
    }
  }
  // No copy may still land in shared memory when the CTA ends (after a
  // timeout or a stop: one more bounded wait each).
  if (tid == 0) {
    if (pending) umma::bar_wait(&M.bar, phase);
    if (pending_in) umma::bar_wait(&M.bar_in, ph_in);
    if (pending_z) umma::bar_wait(&M.bar_z, ph_z);
  }
  __syncthreads();
}

// A bf16 [rows][width] tensor read in boxes of 128 columns x box_rows rows.
bool encode_rows128(CUtensorMap *m, const void *base, long long width, long long rows, int box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)rows, 1};
  const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * rows};
  const cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, bool bf16, cudaStream_t s) {
  if (a.d.T < 1 || a.d.T > kDecodeMaxT) return cudaErrorInvalidValue;
  dim3 grid((unsigned)(a.d.B * a.d.Hv)), block(kThreads);
  const bool raw = a.gate.g == nullptr;
  if (a.d.T == 1 && !a.S_snap) {
    if (bf16)
      (raw ? decode1_kernel<__nv_bfloat16, true> : decode1_kernel<__nv_bfloat16, false>)<<<grid, block, 0, s>>>(a);
    else
      (raw ? decode1_kernel<float, true> : decode1_kernel<float, false>)<<<grid, block, 0, s>>>(a);
  } else {
    auto kern = bf16 ? (raw ? decode_kernel<__nv_bfloat16, true> : decode_kernel<__nv_bfloat16, false>)
                     : (raw ? decode_kernel<float, true> : decode_kernel<float, false>);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecodeSmem);
    if (e != cudaSuccess) return e;
    const long long units = (long long)a.d.B * a.d.Hv;
    const unsigned g = (unsigned)(units < 2LL * sms ? units : 2LL * sms);  // two resident CTAs per SM
    CUtensorMap tm_x{}, tm_w{}, tm_z{};
    if (bf16) {
      const long long C = a.d.C, rows = (long long)a.d.B * a.d.T;
      if (!encode_rows128(&tm_x, a.qkv_pre, C, rows, a.d.T) || !encode_rows128(&tm_w, a.conv_in, C, 3LL * a.d.B, 3) ||
          !encode_rows128(&tm_z, a.z, (long long)a.d.Hv * kD, rows, a.d.T))
        return cudaErrorInvalidValue;
    }
    kern<<<g, block, kDecodeSmem, s>>>(a, tm_x, tm_w, tm_z);
  }
  return cudaGetLastError();
}

}  // namespace gdn
