// chunk_math.cuh -- device pieces of the chunked (WY) form shared by the
// chunk-parallel prefill kernels (prefill_split.cu): the chunk's gate vectors,
// fp16 operand packing, the blocked triangular inverse, and the TMA store /
// named-barrier wrappers.
//
// Page "How Qwen3.5 works" (azmle112.github.io), section 9.11: for a chunk of
// n = 64 tokens, d_i = prod_{r<=i} alpha_r, A = I + tril((B K K^T) o R, -1)
// with R_ij = d_i / d_j, and T = A^{-1} gives U = T B V and W = T B D K.
// Decay ratios are formed from differences of chunk-local cumulative log
// decays G (G_i = sum_{r<=i} g_r), never as a quotient of two small products;
// g is clamped at kGMin.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "launch.h"
#include "umma.cuh"

namespace gdn {
namespace chunk {

using namespace umma;

constexpr int kC = 64;            // chunk length
constexpr float kGMin = -80.0f;   // log-decay clamp (e^-80 ~ 1.8e-35)
constexpr int kLs = 68;           // padded row stride (floats) of the fp32 L scratch

// ---- named barriers -------------------------------------------------------
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// bar.red.or over the named barrier's threads: true if any thread passed true.
__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, t;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred t, %2, %3, q;\n\tselp.u32 %0, 1, 0, t;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---- TMA stores (shared -> global), bulk groups ---------------------------
__device__ __forceinline__ void tma_store_2d(const void *map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, int c0, int c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared-memory sources of this thread's committed stores may be reused.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// This thread's committed stores are complete (visible in global memory).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// ... all but the most recently committed group.
__device__ __forceinline__ void bulk_wait_all_but_one() { asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); }

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes (raw words), no
// wait: tmem_wait_ld() before the registers are used.
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// ---- small arithmetic ------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// silu(x) = x / (1 + 2^(-x log2 e)), on one ex2 and one rcp per value.
__device__ __forceinline__ float silu1(float x) {
  return x * rcp_approx(1.0f + ex2_approx(x * -1.4426950408889634f));
}
// The same for a pair on the paired fp32 pipes.
__device__ __forceinline__ float2 silu2(float2 x) {
  float2 e = __fmul2_rn(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  e = make_float2(ex2_approx(e.x), ex2_approx(e.y));
  float2 dn = __fadd2_rn(e, make_float2(1.0f, 1.0f));
  return __fmul2_rn(x, make_float2(rcp_approx(dn.x), rcp_approx(dn.y)));
}
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// Widen 8 bf16 (one 16-byte chunk) to four channel pairs.
__device__ __forceinline__ void widen(uint4 u, float2 (&v)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

// hi = fp16(v), lo = fp16(v - hi) of a pair, as two packed words, both
// saturated to the finite fp16 range.
__device__ __forceinline__ void split2(float a, float b, uint32_t &whi, uint32_t &wlo) {
  whi = pack2_sat(a, b);
  __half2 th = *reinterpret_cast<__half2 *>(&whi);
  const float2 r = __ffma2_rn(__half22float2(th), make_float2(-1.f, -1.f), make_float2(a, b));
  wlo = pack2_sat(r.x, r.y);
}
// The same for a pair known to lie well inside the fp16 range (no clamp).
__device__ __forceinline__ void split2_inrange(float a, float b, uint32_t &whi, uint32_t &wlo) {
  __half2 th = __floats2half2_rn(a, b);
  const float2 r = __ffma2_rn(__half22float2(th), make_float2(-1.f, -1.f), make_float2(a, b));
  __half2 tl = __floats2half2_rn(r.x, r.y);
  whi = *reinterpret_cast<uint32_t *>(&th);
  wlo = *reinterpret_cast<uint32_t *>(&tl);
}
__device__ __forceinline__ uint32_t pack2_inrange(float a, float b) {
  __half2 t = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&t);
}
// 8 values -> one 16-byte fp16 chunk, no clamp.
__device__ __forceinline__ void st_h8_inrange(uint8_t *p, const float *v) {
  *reinterpret_cast<uint4 *>(p) = make_uint4(pack2_inrange(v[0], v[1]), pack2_inrange(v[2], v[3]),
                                             pack2_inrange(v[4], v[5]), pack2_inrange(v[6], v[7]));
}

// ---- the chunk's gate vectors ---------------------------------------------
struct __align__(16) ChunkVecs {
  float G[kC];     // chunk-local cumulative log decay
  float d[kC];     // e^{G_i}
  float dinv[kC];  // e^{-G_j} (only when the chunk's decay is mild)
  float gam[kC];   // e^{G_last - G_j}
  float beta[kC];
  float bd[kC];    // beta_j d_j
  int mild;        // G_last >= -40: ratios as d_i * dinv_j
};

// g and beta of the chunk's tokens t0 .. t0+63 (one warp: tokens lane and
// lane + 32; the element of token t is (bos + t) Hv + h), as given or as the
// raw projections a, b (their bf16 bits, widened in finish_gb).  Tokens at or
// past T get g = 0, beta = 0.
template <bool kRaw>
__device__ __forceinline__ void load_gb(const GateSrc &gs, long long bos, int Hv, int h, int t0, int T, int lane,
                                        float (&gv)[2], float (&bv)[2]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = t0 + lane + 32 * u;
    gv[u] = 0.f;
    bv[u] = 0.f;
    if (t < T) {
      const long long i = (bos + t) * Hv + h;
      if (kRaw) {
        gv[u] = __uint_as_float(static_cast<const unsigned short *>(gs.a)[i]);
        bv[u] = __uint_as_float(static_cast<const unsigned short *>(gs.b)[i]);
      } else {
        gv[u] = gs.g[i];
        bv[u] = gs.beta[i];
      }
    }
  }
}
// Raw projections -> gates ("How Qwen3.5 works" section 9.5), then the clamp.
template <bool kRaw>
__device__ __forceinline__ void finish_gb(float neg_exp_A, float dt_bias, int t0, int T, int lane, float (&gv)[2],
                                          float (&bv)[2]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (kRaw && t0 + lane + 32 * u < T)
      raw_gate_math(__uint_as_float(__float_as_uint(gv[u]) << 16), __uint_as_float(__float_as_uint(bv[u]) << 16),
                    neg_exp_A, dt_bias, gv[u], bv[u]);
    gv[u] = fmaxf(gv[u], kGMin);
  }
}
// The chunk vectors from its g and beta (one warp); returns e^{G_last}.
__device__ __forceinline__ float chunk_vectors(ChunkVecs &V, float (&gv)[2], const float (&bv)[2], int lane) {
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      float y = __shfl_up_sync(0xffffffffu, gv[u], off);
      if (lane >= off) gv[u] += y;
    }
  gv[1] += __shfl_sync(0xffffffffu, gv[0], 31);
  const float Glast = __shfl_sync(0xffffffffu, gv[1], 31);
  const bool mild = Glast >= -40.f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = lane + 32 * u;
    V.G[i] = gv[u];
    const float di = __expf(gv[u]);
    V.d[i] = di;
    V.dinv[i] = mild ? __expf(-gv[u]) : 0.f;
    V.gam[i] = __expf(Glast - gv[u]);
    V.beta[i] = bv[u];
    V.bd[i] = bv[u] * di;
  }
  if (lane == 0) V.mild = mild ? 1 : 0;
  return __expf(Glast);
}

// ---- the triangular inverse -------------------------------------------------
// Where the solve reads and writes (shared memory): L fp32 [64][kLs] (strictly
// lower, decayed beta K K^T), the fp32 T scratch [64][64] (swizzled, tfi),
// the block-product scratch P (4 KB), and the fp16 K-major [i][j] 64 x 64
// tiles T diag(beta) hi and lo and -T diag(beta d).
struct SolveSmem {
  const float *L;
  float *Tf;
  float *P;
  uint8_t *tu, *tul, *tw;
};

__device__ __forceinline__ int tfi(int row, int col) {
  return row * kC + ((((col >> 2) ^ (row & 15)) << 2) | (col & 3));
}
// acc += s t, on the paired fp32 pipes.
__device__ __forceinline__ void fma4(float4 &acc, float s, const float4 t) {
  const float2 ss = make_float2(s, s);
  const float2 lo = __ffma2_rn(ss, make_float2(t.x, t.y), make_float2(acc.x, acc.y));
  const float2 hi = __ffma2_rn(ss, make_float2(t.z, t.w), make_float2(acc.z, acc.w));
  acc = make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Row i, columns j .. j+3 of T -> T diag(beta) (hi, lo) and -T diag(beta d)
// (negated, so that the W product yields -W^T, the operand the Delta product
// takes), one 8-byte store each.
__device__ __forceinline__ void store_T4(const SolveSmem &s, const ChunkVecs &V, int i, int j, float4 t) {
  const float4 b = ld4(V.beta + j), e = ld4(V.bd + j);
  uint32_t hw[2], lw[2], ww[2];
  split2(t.x * b.x, t.y * b.y, hw[0], lw[0]);
  split2(t.z * b.z, t.w * b.w, hw[1], lw[1]);
  ww[0] = pack2_sat(-(t.x * e.x), -(t.y * e.y));
  ww[1] = pack2_sat(-(t.z * e.z), -(t.w * e.w));
  const uint32_t o = kmaj(i, j, kC);
  *reinterpret_cast<uint2 *>(s.tu + o) = make_uint2(hw[0], hw[1]);
  *reinterpret_cast<uint2 *>(s.tul + o) = make_uint2(lw[0], lw[1]);
  *reinterpret_cast<uint2 *>(s.tw + o) = make_uint2(ww[0], ww[1]);
}

// Zero the 16 x 16 blocks above the diagonal of the fp16 T tiles: items
// q0 .. q1-1 of 3 tiles x 6 blocks x 32 (tile 0 = T diag(beta) hi, 1 = lo,
// 2 = -T diag(beta d)), strided by nthreads from `first`.
__device__ __forceinline__ void zero_T_upper(const SolveSmem &s, int first, int nthreads, int q0, int q1) {
  for (int q = q0 + first; q < q1; q += nthreads) {
    const int tile = q / 192, rem = q % 192, blk = rem / 32, w = rem % 32;
    const int I = blk < 3 ? 0 : blk < 5 ? 1 : 2;
    const int J = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
    const int i = 16 * I + (w >> 1), j = 16 * J + 8 * (w & 1);
    uint8_t *t = tile == 0 ? s.tu : tile == 1 ? s.tul : s.tw;
    *reinterpret_cast<uint4 *>(t + kmaj(i, j, kC)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// T = (I + L)^{-1} (L strictly lower, 64 x 64) in fp32 by recursive doubling on
// 16 x 16 blocks, by 256 threads (tid 0..255) that meet on named barrier
// `bar`: the four diagonal blocks by forward substitution (one column per
// thread, tid 0..63, column-oriented over 4-wide column blocks so that the
// dependent chain is short; the other threads call `idle` meanwhile); the 32 x 32
// halves by T_BA = -T_BB (L_BA T_AA); the whole by the same identity on the
// halves.  Threads idle in a product convert finished blocks to the fp16 tiles
// meanwhile.  With zero_upper, threads 128..255 re-zero the upper blocks of
// all three tiles during the last product (for callers that stage other data
// in the tiles' space between solves).
template <typename Idle>
__device__ __forceinline__ void solve_T(const SolveSmem &s, const ChunkVecs &V, int tid, int bar, bool zero_upper,
                                        Idle &&idle) {
  const float *L = s.L;
  float *Tf = s.Tf;
  float *P = s.P;
  if (tid < kC) {
    // x = (I + L_bb)^{-1} e_c: once x_j .. x_j+3 are final, their terms
    // leave every later row at once.
    const int base = 16 * (tid >> 4), c = tid & 15;
    const float *Lb = L + base * kLs + base;
    float xv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) xv[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      const float4 l1 = ld4(Lb + (j + 1) * kLs + j), l2 = ld4(Lb + (j + 2) * kLs + j), l3 = ld4(Lb + (j + 3) * kLs + j);
      xv[j + 1] = fmaf(-l1.x, xv[j], xv[j + 1]);
      xv[j + 2] = fmaf(-l2.y, xv[j + 1], fmaf(-l2.x, xv[j], xv[j + 2]));
      xv[j + 3] = fmaf(-l3.z, xv[j + 2], fmaf(-l3.y, xv[j + 1], fmaf(-l3.x, xv[j], xv[j + 3])));
#pragma unroll
      for (int i = j + 4; i < 16; ++i) {
        const float4 l = ld4(Lb + i * kLs + j);
        xv[i] -= fmaf(l.w, xv[j + 3], fmaf(l.z, xv[j + 2], fmaf(l.y, xv[j + 1], l.x * xv[j])));
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tf[tfi(base + i, base + c)] = xv[i];
  } else {
    idle();
  }
  __syncwarp();
  named_sync(bar, 256);
  const int hh = tid >> 6, r16 = (tid >> 2) & 15, c4 = tid & 3;
  const int A = 2 * hh, Bb = A + 1;
  if (tid < 128) {
    const float *Lr = L + (16 * Bb + r16) * kLs + 16 * A;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
      const float4 l = ld4(Lr + k4);
      const int row = 16 * A + k4, col = 16 * A + 4 * c4;
      fma4(acc, l.x, ld4(Tf + tfi(row + 0, col)));
      fma4(acc, l.y, ld4(Tf + tfi(row + 1, col)));
      fma4(acc, l.z, ld4(Tf + tfi(row + 2, col)));
      fma4(acc, l.w, ld4(Tf + tfi(row + 3, col)));
    }
    *reinterpret_cast<float4 *>(P + hh * 256 + r16 * 16 + 4 * c4) = acc;
  } else {  // the diagonal blocks are final (two items per thread)
#pragma unroll
    for (int q = tid - 128; q < 256; q += 128) {
      const int b = q >> 6, row = 16 * b + ((q >> 2) & 15), col = 16 * b + 4 * (q & 3);
      store_T4(s, V, row, col, ld4(Tf + tfi(row, col)));
    }
  }
  __syncwarp();
  named_sync(bar, 256);
  if (tid < 128) {
    const int row = 16 * Bb + r16;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
      const float4 t = ld4(Tf + tfi(row, 16 * Bb + k4));
      fma4(acc, t.x, ld4(P + hh * 256 + (k4 + 0) * 16 + 4 * c4));
      fma4(acc, t.y, ld4(P + hh * 256 + (k4 + 1) * 16 + 4 * c4));
      fma4(acc, t.z, ld4(P + hh * 256 + (k4 + 2) * 16 + 4 * c4));
      fma4(acc, t.w, ld4(P + hh * 256 + (k4 + 3) * 16 + 4 * c4));
    }
    *reinterpret_cast<float4 *>(Tf + tfi(row, 16 * A + 4 * c4)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncwarp();
  named_sync(bar, 256);
  const int r16b = tid >> 3, col = 4 * (tid & 7);
  if (tid < 128) {
    const float *La = L + (32 + r16b) * kLs, *Lb = L + (48 + r16b) * kLs;
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int k4 = 0; k4 < 32; k4 += 4) {
      if (k4 < 16 && col >= 16) continue;  // T[0:16][16:32] is zero
      const float4 la = ld4(La + k4), lb = ld4(Lb + k4);
      const float4 t0 = ld4(Tf + tfi(k4 + 0, col)), t1 = ld4(Tf + tfi(k4 + 1, col));
      const float4 t2 = ld4(Tf + tfi(k4 + 2, col)), t3 = ld4(Tf + tfi(k4 + 3, col));
      fma4(acc0, la.x, t0);
      fma4(acc1, lb.x, t0);
      fma4(acc0, la.y, t1);
      fma4(acc1, lb.y, t1);
      fma4(acc0, la.z, t2);
      fma4(acc1, lb.z, t2);
      fma4(acc0, la.w, t3);
      fma4(acc1, lb.w, t3);
    }
    *reinterpret_cast<float4 *>(P + r16b * 32 + col) = acc0;
    *reinterpret_cast<float4 *>(P + (16 + r16b) * 32 + col) = acc1;
  } else {  // the blocks T_10 and T_32 are final
    const int q = tid - 128, h2 = q >> 6;
    const int row = 16 * (2 * h2 + 1) + ((q >> 2) & 15), cc = 32 * h2 + 4 * (q & 3);
    store_T4(s, V, row, cc, ld4(Tf + tfi(row, cc)));
  }
  __syncwarp();
  named_sync(bar, 256);
  if (tid < 128) {  // rows 32 + r (16 terms) and 48 + r (32 terms); T[32:48][48:64] is zero
    const int ra = 32 + r16b, rb = 48 + r16b;
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
      const float4 ta = ld4(Tf + tfi(ra, 32 + k4)), tb = ld4(Tf + tfi(rb, 32 + k4));
      const float4 p0 = ld4(P + (k4 + 0) * 32 + col), p1 = ld4(P + (k4 + 1) * 32 + col);
      const float4 p2 = ld4(P + (k4 + 2) * 32 + col), p3 = ld4(P + (k4 + 3) * 32 + col);
      fma4(acc0, ta.x, p0);
      fma4(acc1, tb.x, p0);
      fma4(acc0, ta.y, p1);
      fma4(acc1, tb.y, p1);
      fma4(acc0, ta.z, p2);
      fma4(acc1, tb.z, p2);
      fma4(acc0, ta.w, p3);
      fma4(acc1, tb.w, p3);
    }
#pragma unroll
    for (int k4 = 16; k4 < 32; k4 += 4) {
      const float4 tb = ld4(Tf + tfi(rb, 32 + k4));
      fma4(acc1, tb.x, ld4(P + (k4 + 0) * 32 + col));
      fma4(acc1, tb.y, ld4(P + (k4 + 1) * 32 + col));
      fma4(acc1, tb.z, ld4(P + (k4 + 2) * 32 + col));
      fma4(acc1, tb.w, ld4(P + (k4 + 3) * 32 + col));
    }
    store_T4(s, V, ra, col, make_float4(-acc0.x, -acc0.y, -acc0.z, -acc0.w));
    store_T4(s, V, rb, col, make_float4(-acc1.x, -acc1.y, -acc1.z, -acc1.w));
  } else if (zero_upper) {
    zero_T_upper(s, tid - 128, 128, 0, 3 * 192);
  }
}

// K steps of one MMA family issued by a whole converged warp (lane 0 issues).
template <typename FA, typename FB>
__device__ __forceinline__ void issue_w(uint32_t d, uint32_t id, int nk, bool accumulate_first, FA da, FB db) {
#pragma unroll
  for (int ks = 0; ks < nk; ++ks) mma_w(d, da(ks), db(ks), id, (accumulate_first || ks > 0) ? 1u : 0u);
}
// The same with A in TMEM at column a0 (8 columns per K step of 16 fp16).
template <typename FB>
__device__ __forceinline__ void issue_ta_w(uint32_t d, uint32_t a0, uint32_t id, int nk, bool accumulate_first,
                                           FB db) {
#pragma unroll
  for (int ks = 0; ks < nk; ++ks) mma_ta_w(d, a0 + 8 * ks, db(ks), id, (accumulate_first || ks > 0) ? 1u : 0u);
}

}  // namespace chunk
}  // namespace gdn
