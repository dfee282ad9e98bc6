// prefill_chunked.cu -- the chunked (WY) form of the gated delta rule on the
// tcgen05 tensor cores (bf16 io).
//
// Page "How Qwen3.5 works" (azmle112.github.io), section 9.11, writes one
// chunk of n = 64 tokens with incoming state S (k x v there) as
//   d_i = prod_{r<=i} alpha_r,   R_ij = d_i / d_j (j <= i),
//   A = I + tril((B K K^T) o R, -1),  U = A^{-1} B V,  W = A^{-1} B D K,
//   Delta = U - W S,  O = D Q S + ((Q K^T) o R) Delta,
//   S_out = d_n S + K^T diag(d_n / d_j) Delta.
// This kernel keeps the state value-major (S[v][k], the node gdn.core
// orientation of the Qwen3.8-27B spec), so every state-dependent product has
// the 128 value rows as its M dimension.  With T = A^{-1}:
//   U^T = V^T (T B)^T          W^T = K^T (T B D)^T        (B, B D folded into T)
//   Delta^T = U^T - S W^T      O^T = (S Q^T) D + Delta^T M^T,  M = (Q K^T) o R
//   S_out = d_n S + Delta^T (Gamma K),   Gamma = diag(d_n / d_j)
// Ratios of decays come from differences of chunk-local cumulative log
// decays G (never a division of two small products); g is clamped at -80.
//
// One CTA per (sequence b, value head h), 12 warps, a sequential loop over the
// chunks.  The fp32 state lives in TMEM for the whole sequence; its fp16 copy,
// the MMA operand, lives in TMEM too (tcgen05.mma reads A from TMEM), as do
// the fp16 Delta^T tiles.  The raw q|k|v rows of a chunk (with the three rows
// before it) and its z rows arrive by TMA into shared memory, a chunk ahead.
// All MMA operands are fp16 (11-bit significand; bf16's 8 bits cost several
// percent of the output's rms at the heavy tail of the gated norm) with fp32
// accumulation.  The operands that feed the state, V and T B (through U) and
// both factors of the state update, are carried as hi + lo fp16 pairs (three
// MMAs for hi*hi + hi*lo + lo*hi), which keeps the state within about 1e-3
// of its rms where single fp16 gives 2e-2 on short, heavy-tailed updates.
// Operands derived from the inputs (v, the initial state, T) are saturated to
// the finite fp16 range in the conversion (cvt .satfinite); Gamma k^ and M
// (|.| <= 1), W, the state's fp16 copy and Delta are converted without it, so
// an entry of those beyond 65504 (far outside any model's regime) would
// overflow to inf.
// Per chunk, in order:
//   A  conv + SiLU + L2 norms of q and k (front end) from the staged raw rows
//      (staged path: q^ and k^ come by TMA; only Gamma k^ is formed)
//   B  MMA1  [K;Q] K^T -> K K^T, Q K^T;  MMA5  S Q^T
//   C  decayed lower-triangular L (fp32) and M (fp16)
//   D  T = (I + L)^{-1} in 16 x 16 blocks (fp32, CUDA cores, warps 0-7) ->
//      T B, T B D; meanwhile the v tiles (conv + SiLU of v, warps 8-11)
//   E  MMA2  U^T = V^T (T B)^T (split);  MMA3  -W^T = K^T (-T B D)^T;
//      the next chunk's raw rows are requested (TMA), and its q^ and k^
//   F  -W^T to shared memory
//   G  MMA4  Delta^T = U^T - S W^T
//   H  Delta^T (hi, lo) to TMEM
//   I  MMA6  Delta^T M^T;            MMA7  S += Delta^T (Gamma K) (split)
//   J  O = d (S Q^T) + Delta^T M^T (warps 0-7) and the gated RMSNorm (node
//      gdn.norm) -> o, tokens 0-47 on warps 0-7 and 48-63 on warps 8-11,
//      which first, once MMA7 is done, pass S on (fp16 copy and rescaled
//      state for the next chunk, or S_T after the last); then the next
//      chunk's z rows are requested
// Each MMA group commits to its own mbarrier, so a phase waits only for the
// products it reads (C for K K^T, F for W^T, J for O) while the rest of the
// chain (S Q^T, U^T, the state update) keeps the tensor pipe busy.
#include <cuda.h>

#include "gdn_device.cuh"
#include "launch.h"
#include "tma_host.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;          // chunk length
constexpr int kThreads = 384;   // 12 warps
constexpr int kTmemWarps = 8;   // warps 0..7 do the TMEM <-> register passes (two per lane quadrant)
constexpr float kGMin = -80.0f;
constexpr int kBarTmem = 1;  // named barrier of warps 0-7 in the epilogue
constexpr int kBarMma6 = 2;  // warp 0 (MMA6 issued) -> warp 11 (may issue MMA7)
constexpr int kBarMma3 = 3;  // warp 0 (MMA3 issued) -> warp 11 (may issue MMA2)
constexpr int kBarSolve = 4;  // warps 0-7 in the solve
constexpr int kBarEpi = 5;    // warps 8-11 in the epilogue (the next chunk's decay formed)
constexpr int kBarJ1 = 6;     // warps 0-7 (O staged) -> warps 8-11 (may read it)

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
constexpr int kRawRows = kC + 3;                  // a chunk's rows plus the three before it
constexpr uint32_t kRawBlock = kRawRows * kD * 2;  // one of q | k | v, bytes (17152)

// Shared memory map (byte offsets from a 1024-aligned base).  fp16 tiles.
constexpr uint32_t OFF_KQ = 0;          // [K;Q] K-major, 128 rows x 128       32 KB
constexpr uint32_t OFF_VH = 32768;      // V hi      MN-major [j][v]           16 KB
constexpr uint32_t OFF_VL = 49152;      // V lo                                16 KB
constexpr uint32_t OFF_GK = 65536;      // Gamma K hi  MN-major [j][k]         16 KB (fused path)
constexpr uint32_t OFF_GKL = 81920;     // Gamma K lo                          16 KB (fused path)
constexpr uint32_t OFF_KQ2 = OFF_GK;    // staged path: the second [K;Q] buffer  32 KB
constexpr uint32_t OFF_TU = 98304;      // T diag(beta)      K-major [i][j]     8 KB
constexpr uint32_t OFF_TW = 106496;     // -T diag(beta d)   K-major [i][j]     8 KB
constexpr uint32_t OFF_M = 114688;      // M         K-major [i][j]             8 KB
constexpr uint32_t OFF_NW = 122880;     // -W^T      MN-major [k][i]           16 KB
constexpr uint32_t OFF_TUL = 139264;    // T diag(beta), low part               8 KB
constexpr uint32_t OFF_RAW = 147456;    // raw q | k | v rows, bf16 [3][67][128] 50.25 KB
constexpr uint32_t OFF_Z = OFF_RAW + 3 * kRawBlock;  // z rows, bf16 [64][128]  16 KB
constexpr uint32_t OFF_VEC = OFF_Z + kC * kD * 2;     // per-token vectors, flags, barriers
// Scratch that lives only between two uses of the tiles it overlays:
constexpr int kLs = 68;                              // padded row stride of L (floats)
constexpr uint32_t OFF_L = OFF_RAW;                  // L fp32 [64][68], phases C-D
constexpr uint32_t OFF_TF = OFF_NW;                  // T fp32 [64][64], phase D
constexpr uint32_t OFF_OST = OFF_M;                  // O^T staging fp32 [64][128] (M, NW, TUL), phase J
// staged path: k^ lo, K-major [64][128] fp16, from before MMA7 of the previous
// chunk completes to MMA7 of this one: beside L in the q and k row blocks
constexpr uint32_t OFF_KLO = OFF_L + 64 * kLs * 4;
static_assert(OFF_KLO % 1024 == 0 && OFF_KLO + kC * kD * 2 <= OFF_RAW + 2 * kRawBlock, "L and k^ lo share the q and k row blocks");
static_assert(OFF_KQ2 % 1024 == 0 && OFF_GKL == OFF_GK + 16384, "the second [K;Q] buffer spans Gamma K hi and lo");
static_assert(OFF_NW == OFF_M + 8192 && OFF_TUL == OFF_NW + 16384, "the staging spans M, NW and TUL");
constexpr uint32_t kVecBytes = 3584;
constexpr uint32_t OFF_PB = OFF_VEC + kVecBytes;  // block products fp32 [32][32], phase D
constexpr uint32_t kSmemUsed = OFF_PB + 32 * 32 * 4;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack
static_assert(OFF_RAW % 128 == 0 && OFF_Z % 128 == 0 && kRawBlock % 128 == 0, "TMA destinations");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// TMEM columns (512 allocated).
constexpr uint32_t TM_S = 0;      // state, fp32 [v][k]                         128 columns
constexpr uint32_t TM_O1 = 128;   // S Q^T [v][i]                               64
constexpr uint32_t TM_O2 = 192;   // Delta^T M^T [v][i]                         64
constexpr uint32_t TM_U = 256;    // U^T, then Delta^T [v][j]                   64
constexpr uint32_t TM_W = 320;    // W^T [k][i]                                 64
constexpr uint32_t TM_KQ = 384;   // [K K^T; Q K^T]; then Delta^T fp16 hi | lo  64
constexpr uint32_t TM_S16 = 448;  // state, fp16 pairs [v][k/2]                 64
constexpr uint32_t kTmemCols = 512;

struct __align__(16) ChunkVecs {  // per-token vectors of one chunk
  float G[kC];     // chunk-local cumulative log decay
  float d[kC];     // e^{G_i}
  float dinv[kC];  // e^{-G_j} (only when the chunk's decay is mild)
  float gam[kC];   // e^{G_last - G_j}
  float beta[kC];
  float bd[kC];    // beta_j d_j
  int mild;        // G_last >= -40: ratios as d_i * dinv_j
};
struct __align__(16) Vecs {  // shared-memory scalars, vectors and barriers
  ChunkVecs cv[2];  // chunk n uses cv[n & 1]; chunk n + 1's are formed during chunk n's epilogue
  float dC_next;   // e^{G_last} of the next chunk
  int abort;
  uint32_t tmem;
  uint64_t bar_qk;   // MMA1 done (K K^T, Q K^T)
  uint64_t bar_w;    // MMA3 done (W^T)
  uint64_t bar_d;    // MMA2, MMA4 done (Delta^T)
  uint64_t bar_o;    // MMA5, MMA6 done (S Q^T, Delta^T M^T)
  uint64_t bar_s;    // MMA7 done (state update)
  uint64_t bar_sq;   // MMA5 done (S Q^T), issued by the second issuer
  uint64_t bar_u;    // MMA2 done (U^T), issued by the second issuer
  uint64_t bar_end;  // every MMA of both issuers, before TMEM is freed
  uint64_t bar_raw;  // raw rows landed
  uint64_t bar_z;    // z rows landed
  uint64_t bar_kq[2];  // staged path: q^ and k^ hi landed in [K;Q] buffer 0 / 1
  uint64_t bar_klo;    // staged path: k^ lo landed
};
static_assert(sizeof(Vecs) <= kVecBytes, "vector area");

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
// silu(x) = x / (1 + 2^(-x log2 e)) for a pair, on the paired fp32 pipes plus
// one ex2 and one rcp per value.  x -> -inf gives 2^inf = inf, rcp -> 0, -0.
__device__ __forceinline__ float2 silu2(float2 x) {
  float2 e = __fmul2_rn(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  e = make_float2(ex2_approx(e.x), ex2_approx(e.y));
  float2 dn = __fadd2_rn(e, make_float2(1.0f, 1.0f));
  return __fmul2_rn(x, make_float2(rcp_approx(dn.x), rcp_approx(dn.y)));
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// g and beta of the chunk starting at t0 (one warp: tokens lane, lane + 32),
// loaded a chunk ahead of use (gate element of token t: (bos + t) Hv + h),
// as given or as the raw projections a, b; finish_gb, called once the loads
// have landed, forms the gates from raw values.  Padded tokens get g = 0,
// beta = 0; g is clamped at kGMin.
template <bool kRaw>
__device__ __forceinline__ void load_gb(const GateSrc &gs, long long bos, int Hv, int h, int t0, int T,
                                        int lane, float (&gv)[2], float (&bv)[2]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = t0 + lane + 32 * u;
    gv[u] = 0.f;
    bv[u] = 0.f;
    if (t < T) {
      const long long i = (bos + t) * Hv + h;
      if (kRaw) {  // the raw bf16 bits, widened only in finish_gb (no wait on the load here)
        gv[u] = __uint_as_float(static_cast<const unsigned short *>(gs.a)[i]);
        bv[u] = __uint_as_float(static_cast<const unsigned short *>(gs.b)[i]);
      } else {
        gv[u] = gs.g[i];
        bv[u] = gs.beta[i];
      }
    }
  }
}
template <bool kRaw>
__device__ __forceinline__ void finish_gb(float neg_exp_A, float dt_bias, int t0, int T, int lane,
                                          float (&gv)[2], float (&bv)[2]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (kRaw && t0 + lane + 32 * u < T)
      raw_gate_math(__uint_as_float(__float_as_uint(gv[u]) << 16), __uint_as_float(__float_as_uint(bv[u]) << 16),
                    neg_exp_A, dt_bias, gv[u], bv[u]);
    gv[u] = fmaxf(gv[u], kGMin);
  }
}

// Chunk vectors from the chunk's g and beta (one warp); returns e^{G_last}.
__device__ float chunk_vectors(ChunkVecs &V, float (&gv)[2], const float (&bv)[2], int lane) {
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

// Widen 8 bf16 (one 16-byte chunk) to four channel pairs.
__device__ __forceinline__ void widen(uint4 u, float2 (&v)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

// 8 values held as 4 pairs -> one 16-byte fp16 chunk (no range clamp: the
// caller guarantees finite fp16 range).
__device__ __forceinline__ void st_h8_pairs(uint8_t *p, const float2 (&v)[4]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 t = __floats2half2_rn(v[i].x, v[i].y);
    w[i] = *reinterpret_cast<uint32_t *>(&t);
  }
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
// hi = fp16(v) and lo = fp16(v - hi) of a pair, as two packed words, both
// saturated to the finite fp16 range (an entry beyond it cannot be carried;
// saturation keeps it finite).
__device__ __forceinline__ void split2(float a, float b, uint32_t &whi, uint32_t &wlo) {
  whi = pack2_sat(a, b);
  __half2 th = *reinterpret_cast<__half2 *>(&whi);
  const float2 r = __ffma2_rn(__half22float2(th), make_float2(-1.f, -1.f), make_float2(a, b));  // v - hi
  wlo = pack2_sat(r.x, r.y);
}
// hi/lo of a pair known to lie well inside the fp16 range (no clamp).
__device__ __forceinline__ void split2_inrange(float a, float b, uint32_t &whi, uint32_t &wlo) {
  __half2 th = __floats2half2_rn(a, b);
  const float2 r = __ffma2_rn(__half22float2(th), make_float2(-1.f, -1.f), make_float2(a, b));  // v - hi
  __half2 tl = __floats2half2_rn(r.x, r.y);
  whi = *reinterpret_cast<uint32_t *>(&th);
  wlo = *reinterpret_cast<uint32_t *>(&tl);
}
// A pair packed to fp16 without a clamp (values well inside the range).
__device__ __forceinline__ uint32_t pack2_inrange(float a, float b) {
  __half2 t = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&t);
}
// 8 values -> one 16-byte fp16 chunk, no clamp.
__device__ __forceinline__ void st_h8_inrange(uint8_t *p, const float *v) {
  *reinterpret_cast<uint4 *>(p) = make_uint4(pack2_inrange(v[0], v[1]), pack2_inrange(v[2], v[3]),
                                             pack2_inrange(v[4], v[5]), pack2_inrange(v[6], v[7]));
}
// The same as a hi/lo pair of 16-byte chunks.
template <bool kClamp>
__device__ __forceinline__ void st_h8_split_pairs(uint8_t *phi, uint8_t *plo, const float2 (&v)[4]) {
  uint32_t wh[4], wl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (kClamp)
      split2(v[i].x, v[i].y, wh[i], wl[i]);
    else
      split2_inrange(v[i].x, v[i].y, wh[i], wl[i]);
  }
  *reinterpret_cast<uint4 *>(phi) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
  *reinterpret_cast<uint4 *>(plo) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
}

// One front-end pass: block blk (0 q, 1 k, 2 v) for tokens r0 .. r0+ntok-1 of
// the chunk (row r of a staged block is token t0 - 3 + r), one 8-channel
// group per lane, sliding the conv window over the tokens; the L2 norm sums
// over the 16 lanes of a half-warp, which hold one token's 128 channels.
// Writes: q^ and k^ (fp16) into [K;Q]; Gamma k^ (hi, lo); v (hi, lo).
template <int NTOK>
__device__ __forceinline__ void fe_pass(uint8_t *sm, const ChunkVecs &V, const Dims &d, const bf16 *conv_w, int blk,
                                        long long c, int r0, int t0, int T, int grp) {
  const bool has_norm = blk < 2, has_single = blk < 2, has_split = blk > 0, has_gamma = blk == 1;
  const int row_off = blk == 0 ? 64 : 0;
  const float scale = blk == 0 ? d.q_scale : 1.0f;
  uint8_t *const dhi = sm + (blk == 1 ? OFF_GK : OFF_VH);
  uint8_t *const dlo = sm + (blk == 1 ? OFF_GKL : OFF_VL);
  const uint8_t *raw = sm + OFF_RAW + blk * kRawBlock + 16 * grp;  // + 256 * row
  float2 w[4][4];  // [channel pair][tap]
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 a0 = ld_io4(conv_w + 4 * (c + 2 * i)), a1 = ld_io4(conv_w + 4 * (c + 2 * i + 1));
    w[i][0] = make_float2(a0.x, a1.x);
    w[i][1] = make_float2(a0.y, a1.y);
    w[i][2] = make_float2(a0.z, a1.z);
    w[i][3] = make_float2(a0.w, a1.w);
  }
  float2 x0[4], x1[4], x2[4];
  widen(*reinterpret_cast<const uint4 *>(raw + 256 * (r0 + 0)), x0);
  widen(*reinterpret_cast<const uint4 *>(raw + 256 * (r0 + 1)), x1);
  widen(*reinterpret_cast<const uint4 *>(raw + 256 * (r0 + 2)), x2);
#pragma unroll 4
  for (int tt = 0; tt < NTOK; ++tt) {
    const int row = r0 + tt;  // token index within the chunk
    const int t = t0 + row;
    float2 x3[4], u[4];
    widen(*reinterpret_cast<const uint4 *>(raw + 256 * (row + 3)), x3);
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 acc = __fmul2_rn(w[i][0], x0[i]);
      acc = __ffma2_rn(w[i][1], x1[i], acc);
      acc = __ffma2_rn(w[i][2], x2[i], acc);
      acc = __ffma2_rn(w[i][3], x3[i], acc);
      u[i] = silu2(acc);
      ss2 = __ffma2_rn(u[i], u[i], ss2);
      x0[i] = x1[i];
      x1[i] = x2[i];
      x2[i] = x3[i];
    }
    if (t >= T) {  // padding beyond the sequence
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] = make_float2(0.f, 0.f);
      ss2 = make_float2(0.f, 0.f);
    }
    float ss = ss2.x + ss2.y;
    // sum of squares over the 16 groups of this token: one half-warp
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float f = has_norm ? rsqrtf(ss + d.eps_l2) * scale : 1.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __fmul2_rn(u[i], make_float2(f, f));
    if (has_single) st_h8_pairs(sm + OFF_KQ + kmaj(row_off + row, 8 * grp, 128), u);
    if (has_split) {
      const float gm = has_gamma ? V.gam[row] : 1.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] = __fmul2_rn(u[i], make_float2(gm, gm));
      const uint32_t o = mnmaj(8 * grp, row, kC);
      if (has_gamma)
        st_h8_split_pairs<false>(dhi + o, dlo + o, u);  // |Gamma k^| <= 1
      else
        st_h8_split_pairs<true>(dhi + o, dlo + o, u);
    }
  }
}

// A: front end for one chunk (q and k), from the staged raw rows; the v tiles
// are made during the solve (front_end_v).  Work per token is about 78 (q)
// and 127 (k: norm, single and split outputs) units, so k goes to warps 0-7
// (4 tokens per half-warp), q to warps 8-11 (7 tokens) and the last 8 q
// tokens to warps 0-3 (one per half-warp, before their k): at most 586 units
// per half-warp, against 624 with all of q on warps 8-11.
__device__ void front_end(uint8_t *sm, const ChunkVecs &V, const Dims &d, const bf16 *conv_w, int kh, int t0,
                          int T, int tid) {
  const int warp = tid >> 5, lane = tid & 31, grp = lane & 15;
  const long long cq = (long long)kh * kD + 8 * grp, ck = (long long)d.Hk * kD + (long long)kh * kD + 8 * grp;
  if (warp < 8) {
    if (warp < 4) fe_pass<1>(sm, V, d, conv_w, 0, cq, 56 + 2 * warp + (lane >> 4), t0, T, grp);
    fe_pass<4>(sm, V, d, conv_w, 1, ck, 4 * (2 * warp + (lane >> 4)), t0, T, grp);
  } else {
    fe_pass<7>(sm, V, d, conv_w, 0, cq, 7 * (2 * (warp - 8) + (lane >> 4)), t0, T, grp);
  }
}
// The v tiles of the chunk starting at t0 (warps 8-11, 8 tokens per half-warp).
__device__ void front_end_v(uint8_t *sm, const ChunkVecs &V, const Dims &d, const bf16 *conv_w, int h, int t0,
                            int T, int tid) {
  const int warp = tid >> 5, lane = tid & 31, grp = lane & 15;
  fe_pass<8>(sm, V, d, conv_w, 2, 2LL * d.Hk * kD + (long long)h * kD + 8 * grp, 8 * (2 * (warp - 8) + (lane >> 4)),
             t0, T, grp);
}

// T scratch: fp32 [64][64], float4 groups XOR-swizzled by row, so that reads of
// one row by eight threads (eight rows) and broadcast reads stay conflict free.
__device__ __forceinline__ int tfi(int row, int col) {
  return row * kC + ((((col >> 2) ^ (row & 15)) << 2) | (col & 3));
}
__device__ __forceinline__ void fma4(float4 &acc, float s, const float4 t) {
  acc.x = fmaf(s, t.x, acc.x);
  acc.y = fmaf(s, t.y, acc.y);
  acc.z = fmaf(s, t.z, acc.z);
  acc.w = fmaf(s, t.w, acc.w);
}

// Row i, columns j .. j+3 (j % 4 == 0) of T -> the fp16 K-major tiles
// T diag(beta) (hi, lo) and -T diag(beta d) (negated, so that MMA3 yields
// -W^T, the operand MMA4 wants), one 8-byte store each.
__device__ __forceinline__ void store_T4(uint8_t *sm, const ChunkVecs &V, int i, int j, float4 t) {
  const float4 b = ld4(V.beta + j), e = ld4(V.bd + j);
  uint32_t hw[2], lw[2], ww[2];
  split2(t.x * b.x, t.y * b.y, hw[0], lw[0]);
  split2(t.z * b.z, t.w * b.w, hw[1], lw[1]);
  ww[0] = pack2_sat(-(t.x * e.x), -(t.y * e.y));
  ww[1] = pack2_sat(-(t.z * e.z), -(t.w * e.w));
  const uint32_t o = kmaj(i, j, kC);
  *reinterpret_cast<uint2 *>(sm + OFF_TU + o) = make_uint2(hw[0], hw[1]);
  *reinterpret_cast<uint2 *>(sm + OFF_TUL + o) = make_uint2(lw[0], lw[1]);
  *reinterpret_cast<uint2 *>(sm + OFF_TW + o) = make_uint2(ww[0], ww[1]);
}

// The fp16 T tiles are zero above the block diagonal (16 x 16 blocks) in
// every chunk: written before the first chunk (tiles 0, 1, 2 = T diag(beta)
// hi, lo and T diag(beta d); q0 = 0) and, for tile 1, whose space the O
// staging borrows, again in every solve (q0 = 192, items 192 .. 383).
__device__ void zero_T_upper(uint8_t *sm, int tid, int q0 = 0, int nthreads = kThreads, int q1 = 3 * 6 * 32) {
  for (int q = q0 + tid; q < q1; q += nthreads) {
    const int tile = q / 192, rem = q % 192, blk = rem / 32, w = rem % 32;
    const int I = blk < 3 ? 0 : blk < 5 ? 1 : 2;
    const int J = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
    const int i = 16 * I + (w >> 1), j = 16 * J + 8 * (w & 1);
    const uint32_t off = tile == 0 ? OFF_TU : tile == 1 ? OFF_TUL : OFF_TW;
    *reinterpret_cast<uint4 *>(sm + off + kmaj(i, j, kC)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// D (warps 0-7): T = (I + L)^{-1} (L strictly lower, 64 x 64), fp32, by recursive
// doubling on 16 x 16 blocks: the four diagonal blocks by forward
// substitution (one column per thread); the two 32 x 32 halves by
// T_BA = -T_BB (L_BA T_AA); then the whole by the same identity on the
// 32 x 32 halves.  Threads idle in a product convert the blocks already
// final into the fp16 tiles meanwhile; the last product converts its own.
// L is [64][kLs] (padded rows), T is [64][64] swizzled (tfi); blocks above
// the diagonal of T are never written (and never read).
__device__ void solve_T(uint8_t *sm, const ChunkVecs &V, int tid) {
  const float *L = reinterpret_cast<const float *>(sm + OFF_L);
  float *Tf = reinterpret_cast<float *>(sm + OFF_TF);
  float *P = reinterpret_cast<float *>(sm + OFF_PB);  // [2][16][16], then [32][32]
  if (tid < kC) {
    const int base = 16 * (tid >> 4), c = tid & 15;
    const float *Lb = L + base * kLs + base;
    float xv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) xv[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int j4 = 0; j4 < i; j4 += 4) {
        const float4 l = ld4(Lb + i * kLs + j4);
        a0 = fmaf(l.x, xv[j4], a0);
        if (j4 + 1 < i) a1 = fmaf(l.y, xv[j4 + 1], a1);
        if (j4 + 2 < i) a0 = fmaf(l.z, xv[j4 + 2], a0);
        if (j4 + 3 < i) a1 = fmaf(l.w, xv[j4 + 3], a1);
      }
      xv[i] -= a0 + a1;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tf[tfi(base + i, base + c)] = xv[i];
  }
  __syncwarp();
  named_sync(kBarSolve, kTmemWarps * 32);
  // The 32 x 32 halves (A, B) = (0, 1), (2, 3): P = L_BA T_AA, T_BA = -T_BB P.
  const int h = tid >> 6, r16 = (tid >> 2) & 15, c4 = tid & 3;
  const int A = 2 * h, Bb = A + 1;
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
    *reinterpret_cast<float4 *>(P + h * 256 + r16 * 16 + 4 * c4) = acc;
  } else {  // the diagonal blocks are final (two items per thread)
#pragma unroll
    for (int q = tid - 128; q < 256; q += 128) {
      const int b = q >> 6, row = 16 * b + ((q >> 2) & 15), col = 16 * b + 4 * (q & 3);
      store_T4(sm, V, row, col, ld4(Tf + tfi(row, col)));
    }
  }
  __syncwarp();
  named_sync(kBarSolve, kTmemWarps * 32);
  if (tid < 128) {
    const int row = 16 * Bb + r16;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k4 = 0; k4 < 16; k4 += 4) {
      const float4 t = ld4(Tf + tfi(row, 16 * Bb + k4));
      fma4(acc, t.x, ld4(P + h * 256 + (k4 + 0) * 16 + 4 * c4));
      fma4(acc, t.y, ld4(P + h * 256 + (k4 + 1) * 16 + 4 * c4));
      fma4(acc, t.z, ld4(P + h * 256 + (k4 + 2) * 16 + 4 * c4));
      fma4(acc, t.w, ld4(P + h * 256 + (k4 + 3) * 16 + 4 * c4));
    }
    *reinterpret_cast<float4 *>(Tf + tfi(row, 16 * A + 4 * c4)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncwarp();
  named_sync(kBarSolve, kTmemWarps * 32);
  // The whole: P = L[32:64][0:32] T[0:32][0:32], T[32:64][0:32] = -T[32:64][32:64] P,
  // each thread two rows (r, r + 16) by four columns, so every operand load
  // feeds eight products.
  const int r16b = tid >> 3, col = 4 * (tid & 7);
  if (tid < 128) {
    const float *La = L + (32 + r16b) * kLs, *Lb = L + (48 + r16b) * kLs;
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll 2
    for (int k4 = col >= 16 ? 16 : 0; k4 < 32; k4 += 4) {  // T[0:16][16:32] is zero
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
  } else if (tid < 256) {  // the blocks T_10 and T_32 are final
    const int q = tid - 128, hh = q >> 6;
    const int row = 16 * (2 * hh + 1) + ((q >> 2) & 15), cc = 32 * hh + 4 * (q & 3);
    store_T4(sm, V, row, cc, ld4(Tf + tfi(row, cc)));
  }
  __syncwarp();
  named_sync(kBarSolve, kTmemWarps * 32);
  if (tid < 128) {  // rows 32 + r (T_BB row has 16 terms) and 48 + r (32 terms); T[32:48][48:64] is zero
    const int ra = 32 + r16b, rb = 48 + r16b;
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll 2
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
#pragma unroll 2
    for (int k4 = 16; k4 < 32; k4 += 4) {
      const float4 tb = ld4(Tf + tfi(rb, 32 + k4));
      fma4(acc1, tb.x, ld4(P + (k4 + 0) * 32 + col));
      fma4(acc1, tb.y, ld4(P + (k4 + 1) * 32 + col));
      fma4(acc1, tb.z, ld4(P + (k4 + 2) * 32 + col));
      fma4(acc1, tb.w, ld4(P + (k4 + 3) * 32 + col));
    }
    store_T4(sm, V, ra, col, make_float4(-acc0.x, -acc0.y, -acc0.z, -acc0.w));
    store_T4(sm, V, rb, col, make_float4(-acc1.x, -acc1.y, -acc1.z, -acc1.w));
  } else {
    zero_T_upper(sm, tid - 128, 192, 128, 2 * 192);  // tile 1, overwritten by the O staging
  }
}

// J: the gated RMSNorm (node gdn.norm) of NR tokens i0, i0 + di, ... of the
// chunk, one half-warp per token (8 channels per lane), from the O staging
// and the staged z rows, to o.
template <int NR>
__device__ __forceinline__ void gated_norm(const uint8_t *sm, const bf16 *norm_w, bf16 *o, const Dims &d,
                                           long long bos, int h, int t0, int T, int i0, int di, int lane) {
  const float *ost = reinterpret_cast<const float *>(sm + OFF_OST);
  const int hl = lane & 15;
  float2 wn[4];
  widen(*reinterpret_cast<const uint4 *>(norm_w + 8 * hl), wn);
  const int nv = min(kC, T - t0);
  bf16 *ob = o + ((bos + t0) * d.Hv + h) * kD + 8 * hl;
  const long long ostride = (long long)d.Hv * kD;
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int i = i0 + di * m;
    const bool valid = i < nv;
    float4 o0 = make_float4(0.f, 0.f, 0.f, 0.f), o1 = o0;
    uint4 zr = make_uint4(0u, 0u, 0u, 0u);
    if (valid) {
      o0 = ld4(ost + i * kD + 8 * hl);
      o1 = ld4(ost + i * kD + 8 * hl + 4);
      zr = *reinterpret_cast<const uint4 *>(sm + OFF_Z + i * kD * 2 + 16 * hl);
    }
    float ss = dot4(o0, o0) + dot4(o1, o1);
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rstd = rsqrtf(ss * (1.0f / kD) + d.eps_norm);
    float2 zz[4];
    widen(zr, zz);
    const float2 op[4] = {make_float2(o0.x, o0.y), make_float2(o0.z, o0.w), make_float2(o1.x, o1.y),
                          make_float2(o1.z, o1.w)};
    uint32_t yw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 sg = silu2(zz[q]);
      const float2 y = __fmul2_rn(__fmul2_rn(wn[q], __fmul2_rn(op[q], make_float2(rstd, rstd))), sg);
      __nv_bfloat162 t = __floats2bfloat162_rn(y.x, y.y);
      yw[q] = *reinterpret_cast<uint32_t *>(&t);
    }
    if (valid) *reinterpret_cast<uint4 *>(ob + i * ostride) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
  }
}

// K steps of one MMA family; descriptors built by the caller's lambdas.
template <typename FA, typename FB>
__device__ __forceinline__ void issue(uint32_t d, uint32_t id, int nk, bool accumulate_first, FA da, FB db) {
  for (int ks = 0; ks < nk; ++ks) mma(d, da(ks), db(ks), id, (accumulate_first || ks > 0) ? 1u : 0u);
}
// The same with A in TMEM at column a0 (8 columns per K step).
template <typename FB>
__device__ __forceinline__ void issue_ta(uint32_t d, uint32_t a0, uint32_t id, int nk, bool accumulate_first,
                                         FB db) {
  for (int ks = 0; ks < nk; ++ks) mma_ta(d, a0 + 8 * ks, db(ks), id, (accumulate_first || ks > 0) ? 1u : 0u);
}
// Both, called by a whole converged warp (lane 0 issues).
template <typename FA, typename FB>
__device__ __forceinline__ void issue_w(uint32_t d, uint32_t id, int nk, bool accumulate_first, FA da, FB db) {
#pragma unroll
  for (int ks = 0; ks < nk; ++ks) mma_w(d, da(ks), db(ks), id, (accumulate_first || ks > 0) ? 1u : 0u);
}
template <typename FB>
__device__ __forceinline__ void issue_ta_w(uint32_t d, uint32_t a0, uint32_t id, int nk, bool accumulate_first,
                                           FB db) {
#pragma unroll
  for (int ks = 0; ks < nk; ++ks) mma_ta_w(d, a0 + 8 * ks, db(ks), id, (accumulate_first || ks > 0) ? 1u : 0u);
}

// Pack 32 fp32 values into 16 fp16-pair words (saturated to the fp16 range).
__device__ __forceinline__ void pack_h16(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
  for (int q = 0; q < 16; ++q) w[q] = pack2_sat(v[2 * q], v[2 * q + 1]);
}

template <bool kRawGates, bool kStagedQK>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_chunked_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tm_qkv,
                           const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_qk) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Vecs &V = *reinterpret_cast<Vecs *>(sm + OFF_VEC);
  const Dims d = a.d;
  const int unit = blockIdx.x;
  const int h = unit % d.Hv;
  int b = unit / d.Hv;
  const int r = d.Hv / d.Hk, kh = h / r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long C = d.C;
  if (a.cu_seqlens && d.B <= kLongestFirstMax)  // packed: the longest sequences first
    b = longest_first(a.cu_seqlens, d.B, b, reinterpret_cast<int *>(sm + OFF_RAW));
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
  const bf16 *x = static_cast<const bf16 *>(a.qkv_pre) + bos * C;
  const bf16 *conv0 = a.conv0 ? static_cast<const bf16 *>(a.conv0) + (long long)b * 3 * C : nullptr;
  const bf16 *conv_w = static_cast<const bf16 *>(a.conv_w);
  const long long unit_off = ((long long)b * d.Hv + h) * kD * kD;
  const uint32_t sbase = smem_u32(sm);
  const int cq = kh * kD, ck = d.Hk * kD + kh * kD, cv = 2 * d.Hk * kD + h * kD;

  // One thread: the raw rows t0-3 .. t0+63 of q, k, v (staged path: of v).
  auto request_raw = [&](int t0) {
    const int row = (int)(bos + t0 - 3);
    if (kStagedQK) {
      bar_expect_tx(&V.bar_raw, kRawBlock);
    } else {
      bar_expect_tx(&V.bar_raw, 3 * kRawBlock);
      tma_load_3d(sbase + OFF_RAW + 0 * kRawBlock, &tm_qkv, cq, row, 0, &V.bar_raw);
      tma_load_3d(sbase + OFF_RAW + 1 * kRawBlock, &tm_qkv, ck, row, 0, &V.bar_raw);
    }
    tma_load_3d(sbase + OFF_RAW + 2 * kRawBlock, &tm_qkv, cv, row, 0, &V.bar_raw);
  };
  // Staged path, one thread: q^ (rows 64..127) and k^ hi (rows 0..63) of tokens
  // t0 .. t0+63 straight into [K;Q] buffer `buf`, two 64-column boxes each.
  auto request_kq = [&](int t0, int buf) {
    const uint32_t kqb = sbase + (buf ? OFF_KQ2 : OFF_KQ);
    bar_expect_tx(&V.bar_kq[buf], 2 * kC * kD * 2);
#pragma unroll
    for (int at = 0; at < 2; ++at) {
      tma_load_3d(kqb + at * 16384 + 64 * 128, &tm_qk, kh * kD + 64 * at, (int)(bos + t0), 0, &V.bar_kq[buf]);
      tma_load_3d(kqb + at * 16384, &tm_qk, kh * kD + 64 * at, (int)(bos + t0), 1, &V.bar_kq[buf]);
    }
  };
  // Staged path, one thread: k^ lo of tokens t0 .. t0+63 (two 64-column boxes).
  auto request_klo = [&](int t0) {
    bar_expect_tx(&V.bar_klo, kC * kD * 2);
    tma_load_3d(sbase + OFF_KLO, &tm_qk, kh * kD, (int)(bos + t0), 2, &V.bar_klo);
    tma_load_3d(sbase + OFF_KLO + kC * 128, &tm_qk, kh * kD + 64, (int)(bos + t0), 2, &V.bar_klo);
  };
  auto request_z = [&](int t0) {  // one thread: the z rows t0 .. t0+63 of head h
    bar_expect_tx(&V.bar_z, kC * kD * 2);
    tma_load_3d(sbase + OFF_Z, &tm_z, h * kD, (int)(bos + t0), 0, &V.bar_z);
  };

  // Carried conv window: the last three raw rows of the channels this CTA owns.
  auto write_conv_T = [&]() {
    bf16 *cT = static_cast<bf16 *>(a.conv_T) + (long long)b * 3 * C;
    const bool own_qk = (h % r) == 0;
    for (int idx = tid; idx < 3 * 3 * kD; idx += kThreads) {
      const int e = idx / (3 * kD), rem = idx % (3 * kD), blk = rem / kD, ch = rem % kD;
      if (blk < 2 && !own_qk) continue;
      const long long c = (blk == 0 ? cq : blk == 1 ? ck : cv) + ch;
      const int t = T - 3 + e;
      bf16 val;
      if (t >= 0) val = x[(long long)t * C + c];
      else if (conv0) val = conv0[(long long)(3 + t) * C + c];
      else val = bf16(0.f);
      cT[(long long)e * C + c] = val;
    }
  };
  if (T == 0) {  // an empty packed sequence: state and window pass through
    float4 *dst = reinterpret_cast<float4 *>(a.S_T + unit_off);
    const float4 *src = a.S0 ? reinterpret_cast<const float4 *>(a.S0 + unit_off) : nullptr;
    if (src != dst)
      for (int i = tid; i < kD * kD / 4; i += kThreads) dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    write_conv_T();
    return;
  }

  if (tid == 0) {
    bar_init(&V.bar_qk, 1);
    bar_init(&V.bar_w, 1);
    bar_init(&V.bar_d, 1);
    bar_init(&V.bar_o, 1);
    bar_init(&V.bar_s, 1);
    bar_init(&V.bar_sq, 1);
    bar_init(&V.bar_u, 1);
    bar_init(&V.bar_end, 2);
    bar_init(&V.bar_raw, 1);
    bar_init(&V.bar_z, 1);
    bar_init(&V.bar_kq[0], 1);
    bar_init(&V.bar_kq[1], 1);
    bar_init(&V.bar_klo, 1);
    V.abort = 0;
  }
  if (warp == 0) tmem_alloc(&V.tmem, kTmemCols);
  zero_T_upper(sm, tid);
  float g_cur[2], b_cur[2], g_nxt[2] = {0.f, 0.f}, b_nxt[2] = {0.f, 0.f};  // warp 11: this and the next chunk
  float neg_exp_A = 0.f, dt_bias = 0.f;          // warp 11, raw gates: -exp(A_log[h]), dt_bias[h]
  if (warp == 11) {
    load_gb<kRawGates>(a.gate, bos, d.Hv, h, 0, T, lane, g_cur, b_cur);
    if (kRawGates) {
      neg_exp_A = -expf(a.gate.A_log[h]);
      dt_bias = a.gate.dt_bias[h];
    }
    finish_gb<kRawGates>(neg_exp_A, dt_bias, 0, T, lane, g_cur, b_cur);
    const float dc0 = chunk_vectors(V.cv[0], g_cur, b_cur, lane);
    if (lane == 0) V.dC_next = dc0;
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (tid == 0) {
    request_raw(0);
    if (kStagedQK) {
      request_kq(0, 0);
      if (T > kC) request_kq(kC, 1);
      request_klo(0);
    }
    request_z(0);
  }
  // Staged path: [K;Q] buffer and k^ lo copies requested and consumed so far
  // (chunk n reads buffer n & 1, its (n >> 1)-th use; k^ lo's n-th use).
  int kq_next = kStagedQK ? (T > kC ? 2 : 1) : 0, kq_used = 0;
  int klo_next = kStagedQK ? 1 : 0, klo_used = 0;
  const uint32_t tmem = V.tmem;
  // TMEM lane quadrant and column half of this warp for the 32x32b accesses.
  const int quad = warp & 3, half = warp >> 2;
  const int lrow = 32 * quad + lane;  // TMEM lane (row) this thread reads
  const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);

  // Initial state: TMEM fp32 <- dC(chunk 0) * S0, TMEM fp16 copy <- S0.
  if (warp < kTmemWarps) {
    const float dc0 = V.dC_next;
    float v[32];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int k0 = 64 * half + 32 * p;
      if (a.S0) {
        const float4 *src = reinterpret_cast<const float4 *>(a.S0 + unit_off + (long long)lrow * kD + k0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 f = src[q];
          v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = 0.f;
      }
      uint32_t w16[16];
      pack_h16(v, w16);
      tmem_st16w(tl + TM_S16 + k0 / 2, w16);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] *= dc0;
      tmem_st32(tl + TM_S + k0, v);
    }
  }

  // Each mbarrier completes once per chunk; its phase bit is tracked here.
  uint32_t ph_qk = 0, ph_w = 0, ph_d = 0, ph_o = 0, ph_s = 0, ph_sq = 0, ph_u = 0, phase_raw = 0, phase_z = 0;
  // MMAs off the critical path are issued by warp 11 (its lane 0), idle in the
  // phases where it issues them; the critical ones by warp 0 (thread 0).  A
  // whole converged warp runs the issue code.  Warp 10 (lane 0) requests the
  // raw rows and the staged q^ / k^ of the next chunk.
  const bool issuer2 = tid == kThreads - 32;
  const bool loader = tid == kThreads - 64;
  bool raw_pending = true, z_pending = true;  // a requested TMA not yet consumed
  const int nchunks = (T + kC - 1) / kC;
  const uint32_t id_kk = idesc(128, 64, 0, 0);
  const uint32_t id_mk = idesc(128, 64, 1, 0);
  const uint32_t id_km = idesc(128, 64, 0, 1);
  const uint32_t id_km128 = idesc(128, 128, 0, 1);

  // All threads: wait on an mbarrier phase; a uniform decision to abort.
  // ok_in: an earlier wait of this thread that is voted on here too.
  auto wait_all = [&](uint64_t *bar, uint32_t &ph, bool ok_in = true) -> bool {
    // Reconverge first: lane 0 of warp 0 issues the MMAs and TMA copies, and
    // while its 31 sibling lanes sat in the polling loop (each try_wait may
    // suspend the warp for a while) that lane lost about a microsecond.
    __syncwarp();
    bool ok = bar_wait(bar, ph);
    ph ^= 1u;
    fence_after();
    const int bad = __syncthreads_or(!(ok && ok_in));
    if (bad && tid == 0) {
      atomicOr(a.err, kErrTimeout);
      V.abort = 1;
    }
    return !bad;
  };
  // Warps 0-7 only (named barrier kBarTmem, 256 threads): wait on an mbarrier
  // phase; a timeout sets the abort flag, seen by all at the end of the chunk.
  auto wait_tmem = [&](uint64_t *bar, uint32_t &ph) -> bool {
    __syncwarp();
    const bool ok = bar_wait(bar, ph);
    ph ^= 1u;
    fence_after();
    __syncwarp();  // the barrier instruction wants the warp converged
    const bool bad = named_sync_or(kBarTmem, kTmemWarps * 32, !ok);
    if (bad && tid == 0) {
      atomicOr(a.err, kErrTimeout);
      V.abort = 1;
    }
    return !bad;
  };
  auto smem_ready = [&]() {  // operands written (shared memory or TMEM) -> visible to the MMA unit
    fence_smem_to_async();
    fence_before();
    __syncthreads();
  };

  for (int n = 0; n < nchunks; ++n) {
    const int t0 = n * kC;
    // A0: chunk vectors; the next chunk's g and beta requested
    ChunkVecs &CV = V.cv[n & 1];  // formed before the loop or during the previous chunk's epilogue
    if (warp == 11 && n + 1 < nchunks) load_gb<kRawGates>(a.gate, bos, d.Hv, h, t0 + kC, T, lane, g_nxt, b_nxt);
    // This chunk's staged rows (fused path: every warp; staged path: warps
    // 8-11, which read only the v rows, while warp 0 waits for q^ and k^ hi
    // in [K;Q]): each warp waits itself (the previous chunk ended on a
    // barrier); a timeout is voted on at the next barrier.
    const uint32_t kqb = sbase + ((kStagedQK && (n & 1)) ? OFF_KQ2 : OFF_KQ);  // this chunk's [K;Q]
    bool start_ok = true;
    __syncwarp();
    if (!kStagedQK || warp >= kTmemWarps) start_ok = bar_wait(&V.bar_raw, phase_raw);
    if (kStagedQK && warp == 0) start_ok = bar_wait(&V.bar_kq[n & 1], (uint32_t)(n >> 1) & 1u);
    phase_raw ^= 1u;
    raw_pending = false;
    if (kStagedQK) {
      ++kq_used;
      // the other buffer's last readers (the previous chunk's MMAs) are done:
      // the next chunk's q^ and k^ may land there
      if (n >= 1 && n + 1 < nchunks) {
        if (loader) request_kq(t0 + kC, (n + 1) & 1);
        ++kq_next;
      }
      if (!start_ok) {  // no barrier votes here: the abort flag is read after F
        atomicOr(a.err, kErrTimeout);
        V.abort = 1;
      }
    }
    if (n == 0) {  // rows before the first token: the carried window, or zeros
      if (!kStagedQK || warp >= kTmemWarps) {  // staged path: the v rows, by warps 8-11 (they waited)
        const int i0 = kStagedQK ? 2 * 48 + tid - kTmemWarps * 32 : tid;
        const int nth = kStagedQK ? kThreads - kTmemWarps * 32 : kThreads;
        for (int idx = i0; idx < 3 * 3 * 16; idx += nth) {
          const int blk = idx / 48, rw = (idx / 16) % 3, g8 = idx % 16;
          const int cc = blk == 0 ? cq : blk == 1 ? ck : cv;
          *reinterpret_cast<uint4 *>(sm + OFF_RAW + blk * kRawBlock + 256 * rw + 16 * g8) =
              conv0 ? *reinterpret_cast<const uint4 *>(conv0 + (long long)rw * C + cc + 8 * g8)
                    : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncthreads();
    }
    auto issue_mma1 = [&]() {  // B: MMA1  [K;Q] K^T (warp 0)
      __syncwarp();
      fence_after();
      issue_w(tmem + TM_KQ, id_kk, 8, false, [&](int ks) { return desc_k(kqb, ks, 128); },
              [&](int ks) { return desc_k(kqb, ks, 128); });
      commit_w(&V.bar_qk);
    };
    // MMA5 S Q^T (Q^ = rows 64..127 of [K;Q], S from TMEM), needed only in J
    auto issue_mma5 = [&]() {
      fence_after();
      issue_ta_w(tmem + TM_O1, tmem + TM_S16, id_kk, 8, false, [&](int ks) { return desc_k(kqb + 64 * 128, ks, 128); });
      commit_w(&V.bar_sq);
    };
    if (kStagedQK) {
      // [K;Q] arrived by TMA: warp 0 issues MMA1 and MMA5 behind it; warps
      // 0-7 wait for MMA1 alone, warps 8-11 go on to the v tiles.
      if (warp == 0) {
        issue_mma1();
        issue_mma5();
      }
      if (warp < kTmemWarps) wait_tmem(&V.bar_qk, ph_qk);  // a timeout sets the abort flag, read after F
      else ph_qk ^= 1u;
    } else {
      // A: front end
      front_end(sm, CV, d, conv_w, kh, t0, T, tid);
      smem_ready();
      if (warp == 0) issue_mma1();
      if (!wait_all(&V.bar_qk, ph_qk, start_ok)) break;
      if (warp == 11) issue_mma5();
    }
    // C: L (fp32, strictly lower, decayed beta K K^T) and M (fp16, decayed Q K^T incl. diagonal)
    if (warp < kTmemWarps) {
      float v[32], rr[32];
      tmem_ld32(tl + TM_KQ + 32 * half, v);
      const int j0 = 32 * half;
      const int i = lrow < kC ? lrow : lrow - kC;
      if (CV.mild) {
        const float di = CV.d[i];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 dv = ld4(CV.dinv + j0 + q);
          const float2 r01 = __fmul2_rn(make_float2(di, di), make_float2(dv.x, dv.y));
          const float2 r23 = __fmul2_rn(make_float2(di, di), make_float2(dv.z, dv.w));
          rr[q] = r01.x;
          rr[q + 1] = r01.y;
          rr[q + 2] = r23.x;
          rr[q + 3] = r23.y;
        }
      } else {
        const float gi = CV.G[i];
#pragma unroll
        for (int q = 0; q < 32; ++q) rr[q] = __expf(gi - CV.G[j0 + q]);
      }
      if (lrow < kC) {
        const float bi = CV.beta[i];
        float *L = reinterpret_cast<float *>(sm + OFF_L) + i * kLs + j0;
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float2 p01 = __fmul2_rn(__fmul2_rn(make_float2(bi, bi), make_float2(v[q], v[q + 1])),
                                        make_float2(rr[q], rr[q + 1]));
          const float2 p23 = __fmul2_rn(__fmul2_rn(make_float2(bi, bi), make_float2(v[q + 2], v[q + 3])),
                                        make_float2(rr[q + 2], rr[q + 3]));
          float4 f;
          f.x = (j0 + q + 0 < i) ? p01.x : 0.f;
          f.y = (j0 + q + 1 < i) ? p01.y : 0.f;
          f.z = (j0 + q + 2 < i) ? p23.x : 0.f;
          f.w = (j0 + q + 3 < i) ? p23.y : 0.f;
          *reinterpret_cast<float4 *>(L + q) = f;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 32; q += 2) {
          const float2 p = __fmul2_rn(make_float2(v[q], v[q + 1]), make_float2(rr[q], rr[q + 1]));
          v[q] = (j0 + q <= i) ? p.x : 0.f;
          v[q + 1] = (j0 + q + 1 <= i) ? p.y : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) st_h8_inrange(sm + OFF_M + kmaj(i, j0 + 8 * q, kC), v + 8 * q);  // |M| <= q_scale
      }
      __syncwarp();
      named_sync(kBarSolve, kTmemWarps * 32);  // L written: the solve may read it (warps 8-11 go on)
    }
    // D: the triangular inverse, scaled copies T B and T B D (warps 0-7);
    // warps 8-11 make this chunk's v tiles from its staged rows meanwhile,
    // from the end of B on (the V tiles were last read by MMA2 of the previous
    // chunk; the raw v rows do not share space with the solve's scratch).
    if (warp < kTmemWarps)
      solve_T(sm, CV, tid);
    else
      front_end_v(sm, CV, d, conv_w, h, t0, T, tid);
    smem_ready();
    // E: MMA2 U^T = V^T (T B)^T, hi*hi + lo*hi + hi*lo; MMA3 -W^T = K^T (-T B D)^T
    // (K^ read from [K;Q] as an MN-major operand).  The raw rows are free now:
    // the loader requests the next chunk's.
    if (n + 1 < nchunks) raw_pending = true;
    if (warp < kTmemWarps) {
      if (warp == 0) {
        fence_after();
        issue_w(tmem + TM_W, id_mk, 4, false,
                [&](int ks) { return desc(kqb + (uint32_t)(ks * 2048), 128 * 128, 1024); },
                [&](int ks) { return desc_k(sbase + OFF_TW, ks, kC); });
        commit_w(&V.bar_w);
        __syncwarp();
        named_arrive(kBarMma3, 64);
      }
      // F: -W^T (lanes k, columns i; the sign comes from the T tile) -> MN-major [k][i]
      if (wait_tmem(&V.bar_w, ph_w)) {
        float v[32];
        tmem_ld32(tl + TM_W + 32 * half, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) st_h8_inrange(sm + OFF_NW + mnmaj(32 * half + 8 * q, lrow, kD), v + 8 * q);
      }
    } else {
      // MMA2 U^T, needed only by MMA4: issued behind MMA3 while F runs
      if (warp == 11) {
        __syncwarp();
        named_sync(kBarMma3, 64);
        fence_after();
        auto a_vh = [&](int ks) { return desc_mn(sbase + OFF_VH, ks, kC); };
        auto b_tu = [&](int ks) { return desc_k(sbase + OFF_TU, ks, kC); };
        issue_w(tmem + TM_U, id_mk, 4, false, a_vh, b_tu);
        issue_w(tmem + TM_U, id_mk, 4, true, [&](int ks) { return desc_mn(sbase + OFF_VL, ks, kC); }, b_tu);
        issue_w(tmem + TM_U, id_mk, 4, true, a_vh, [&](int ks) { return desc_k(sbase + OFF_TUL, ks, kC); });
        commit_w(&V.bar_u);
      }
      if (loader && n + 1 < nchunks) request_raw(t0 + kC);
      ph_w ^= 1u;
    }
    smem_ready();
    if (V.abort) break;
    // G: MMA4 Delta^T = U^T - S W^T (S from TMEM), after MMA2 (the other issuer)
    if (warp == 0) {
      bar_wait(&V.bar_u, ph_u);  // bounded; a stall here ends in the timeout below
      __syncwarp();
      fence_after();
      issue_ta_w(tmem + TM_U, tmem + TM_S16, id_km, 8, true, [&](int ks) { return desc_mn(sbase + OFF_NW, ks, kD); });
      commit_w(&V.bar_d);
    }
    ph_u ^= 1u;
    if (!wait_all(&V.bar_d, ph_d)) break;
    // H: Delta^T (lanes v, columns j) -> fp16 hi and lo pairs in TMEM; in the
    // staged path also (Delta Gamma)^T, the state update's A operand (W^T's
    // columns are free since F), so that MMA7 reads k^ straight from its tiles
    if (warp < kTmemWarps) {
      float v[32];
      tmem_ld32(tl + TM_U + 32 * half, v);
      uint32_t wh[16], wl[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) split2_inrange(v[2 * q], v[2 * q + 1], wh[q], wl[q]);
      tmem_st16w_nw(tl + TM_KQ + 16 * half, wh);
      tmem_st16w_nw(tl + TM_KQ + 32 + 16 * half, wl);
      if (kStagedQK) {
#pragma unroll
        for (int q = 0; q < 32; q += 4) {  // column j = 32 half + q: times e^{G_last - G_j} <= 1
          const float4 g = ld4(CV.gam + 32 * half + q);
          const float2 p01 = __fmul2_rn(make_float2(v[q], v[q + 1]), make_float2(g.x, g.y));
          const float2 p23 = __fmul2_rn(make_float2(v[q + 2], v[q + 3]), make_float2(g.z, g.w));
          v[q] = p01.x;
          v[q + 1] = p01.y;
          v[q + 2] = p23.x;
          v[q + 3] = p23.y;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) split2_inrange(v[2 * q], v[2 * q + 1], wh[q], wl[q]);
        tmem_st16w_nw(tl + TM_W + 16 * half, wh);
        tmem_st16w_nw(tl + TM_W + 32 + 16 * half, wl);
      }
      tmem_wait_st();
    }
    smem_ready();
    // The epilogue.  Warps 0-7 (TMEM) form and store the output and sync
    // among themselves (named barrier 1); warps 8-11 meanwhile issue the state
    // update, pass the state on and take the last 16 tokens of the gated norm.
    // Everyone meets at the end of the chunk.
    if (warp < kTmemWarps) {
      bool ok = true;
      // I: MMA6 Delta^T M^T (warp 0); then warp 11 may issue MMA7 behind it
      if (warp == 0) {
        bar_wait(&V.bar_sq, ph_sq);  // MMA5 (the other issuer) done, so bar_o covers O1 and O2
        __syncwarp();
        fence_after();
        issue_ta_w(tmem + TM_O2, tmem + TM_KQ, id_kk, 4, false, [&](int ks) { return desc_k(sbase + OFF_M, ks, kC); });
        commit_w(&V.bar_o);
        __syncwarp();
        named_arrive(kBarMma6, 64);
      }
      ok = wait_tmem(&V.bar_o, ph_o);
      if (ok) {
      // J1: O^T = d (S Q^T) + Delta^T M^T -> staging [i][v]
        {
        float *ost = reinterpret_cast<float *>(sm + OFF_OST);
        uint32_t ra[32], rb[32];
        tmem_ld32_nw(tl + TM_O1 + 32 * half, ra);
        tmem_ld32_nw(tl + TM_O2 + 32 * half, rb);
        tmem_wait_ld();
        float v[32], w2[32];
  #pragma unroll
        for (int q = 0; q < 32; ++q) {
          v[q] = __uint_as_float(ra[q]);
          w2[q] = __uint_as_float(rb[q]);
        }
  #pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 dq = ld4(CV.d + 32 * half + q);
          const float2 o01 = __ffma2_rn(make_float2(dq.x, dq.y), make_float2(v[q], v[q + 1]), make_float2(w2[q], w2[q + 1]));
          const float2 o23 = __ffma2_rn(make_float2(dq.z, dq.w), make_float2(v[q + 2], v[q + 3]),
                                        make_float2(w2[q + 2], w2[q + 3]));
          ost[(32 * half + q + 0) * kD + lrow] = o01.x;
          ost[(32 * half + q + 1) * kD + lrow] = o01.y;
          ost[(32 * half + q + 2) * kD + lrow] = o23.x;
          ost[(32 * half + q + 3) * kD + lrow] = o23.y;
        }
      }
      }
      __syncwarp();
      named_arrive(kBarJ1, kThreads);  // the O staging is written
      ok = wait_tmem(&V.bar_z, phase_z) && ok;
      z_pending = false;
      if (ok) {
      // J2: gated RMSNorm of tokens 0-47 (warps 0-7; 48-63 on warps 8-11)
      gated_norm<3>(sm, static_cast<const bf16 *>(a.norm_w), static_cast<bf16 *>(a.o), d, bos, h, t0, T,
                    2 * warp + (lane >> 4), 16, lane);
      }
      ph_s ^= 1u;
    } else {
      // MMA7 S += Delta^T (Gamma K), hi*hi + hi*lo + lo*hi, issued once MMA6 is
      // in the queue ahead of it; while it runs, warp 11 forms the next
      // chunk's gates and chunk vectors (through shared memory).
      if (warp == 11) {
        __syncwarp();
        named_sync(kBarMma6, 64);
        if (kStagedQK) {  // this chunk's k^ lo (requested once the previous MMA7 was done)
          if (!bar_wait(&V.bar_klo, (uint32_t)n & 1u) && lane == 0) {
            atomicOr(a.err, kErrTimeout);
            V.abort = 1;
          }
          __syncwarp();
        }
        fence_after();
        if (kStagedQK) {  // S += (Delta Gamma)^T K: A from TMEM (W^T's columns), k^ hi in [K;Q], k^ lo staged
          auto b_kh = [&](int ks) { return desc(kqb + (uint32_t)(ks * 2048), 128 * 128, 1024); };
          issue_ta_w(tmem + TM_S, tmem + TM_W, id_km128, 4, true, b_kh);
          issue_ta_w(tmem + TM_S, tmem + TM_W, id_km128, 4, true,
                     [&](int ks) { return desc(sbase + OFF_KLO + (uint32_t)(ks * 2048), kC * 128, 1024); });
          issue_ta_w(tmem + TM_S, tmem + TM_W + 32, id_km128, 4, true, b_kh);
        } else {
          auto b_gk = [&](int ks) { return desc_mn(sbase + OFF_GK, ks, kC); };
          issue_ta_w(tmem + TM_S, tmem + TM_KQ, id_km128, 4, true, b_gk);
          issue_ta_w(tmem + TM_S, tmem + TM_KQ, id_km128, 4, true,
                     [&](int ks) { return desc_mn(sbase + OFF_GKL, ks, kC); });
          issue_ta_w(tmem + TM_S, tmem + TM_KQ + 32, id_km128, 4, true, b_gk);
        }
        commit_w(&V.bar_s);
        if (n + 1 < nchunks) {
          finish_gb<kRawGates>(neg_exp_A, dt_bias, t0 + kC, T, lane, g_nxt, b_nxt);
          const float dcn = chunk_vectors(V.cv[(n + 1) & 1], g_nxt, b_nxt, lane);
          if (lane == 0) V.dC_next = dcn;
        }
      }
      ph_o ^= 1u;
      // J3 (warps 8-11, all 128 state columns each, alongside J2 on warps
      // 0-7): S -> fp16 copy and rescaled state (or S_T after the last
      // chunk), in TMEM
      __syncwarp();
      named_sync(kBarEpi, 128);  // the next chunk's total decay is formed
      bool ok = bar_wait(&V.bar_s, ph_s);
      ph_s ^= 1u;
      fence_after();
      // MMA7 is done with k^ lo (staged path): the next chunk's may land
      if (kStagedQK && loader && ok && n + 1 < nchunks) request_klo(t0 + kC);
      if (__all_sync(0xffffffffu, ok)) {
        const bool last = n + 1 == nchunks;
        const float dcn = V.dC_next;
#pragma unroll 1
        for (int k0 = 0; k0 < kD; k0 += 64) {
          uint32_t r0[32], r1[32];
          tmem_ld32_nw(tl + TM_S + k0, r0);
          tmem_ld32_nw(tl + TM_S + k0 + 32, r1);
          tmem_wait_ld();
          if (last) {
            float4 *dst = reinterpret_cast<float4 *>(a.S_T + unit_off + (long long)lrow * kD + k0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1]),
                                   __uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3]));
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[8 + q] = make_float4(__uint_as_float(r1[4 * q]), __uint_as_float(r1[4 * q + 1]),
                                       __uint_as_float(r1[4 * q + 2]), __uint_as_float(r1[4 * q + 3]));
          } else {
            uint32_t w16[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) w16[q] = pack2_inrange(__uint_as_float(r0[2 * q]), __uint_as_float(r0[2 * q + 1]));
            tmem_st16w_nw(tl + TM_S16 + k0 / 2, w16);
#pragma unroll
            for (int q = 0; q < 16; ++q) w16[q] = pack2_inrange(__uint_as_float(r1[2 * q]), __uint_as_float(r1[2 * q + 1]));
            tmem_st16w_nw(tl + TM_S16 + k0 / 2 + 16, w16);
#pragma unroll
            for (int q = 0; q < 32; q += 2) {  // paired fp32 multiplies
              float2 x0 = __fmul2_rn(make_float2(__uint_as_float(r0[q]), __uint_as_float(r0[q + 1])), make_float2(dcn, dcn));
              float2 x1 = __fmul2_rn(make_float2(__uint_as_float(r1[q]), __uint_as_float(r1[q + 1])), make_float2(dcn, dcn));
              r0[q] = __float_as_uint(x0.x);
              r0[q + 1] = __float_as_uint(x0.y);
              r1[q] = __float_as_uint(x1.x);
              r1[q + 1] = __float_as_uint(x1.y);
            }
            tmem_st32w_nw(tl + TM_S + k0, r0);
            tmem_st32w_nw(tl + TM_S + k0 + 32, r1);
            tmem_wait_st();
          }
        }
      } else if (lane == 0) {
        atomicOr(a.err, kErrTimeout);
        V.abort = 1;
      }
      // J2 of tokens 48-63, once warps 0-7 have staged O and the z rows landed
      __syncwarp();
      named_sync(kBarJ1, kThreads);
      const bool zok = bar_wait(&V.bar_z, phase_z);
      phase_z ^= 1u;
      if (__all_sync(0xffffffffu, zok)) {
        gated_norm<2>(sm, static_cast<const bf16 *>(a.norm_w), static_cast<bf16 *>(a.o), d, bos, h, t0, T,
                      48 + 2 * (warp - 8) + (lane >> 4), 8, lane);
      } else if (lane == 0) {
        atomicOr(a.err, kErrTimeout);
        V.abort = 1;
      }
    }
    ph_sq ^= 1u;
    if (kStagedQK) {
      ++klo_used;
      if (n + 1 < nchunks) ++klo_next;
    }
    fence_before();
    fence_smem_to_async();  // z, the staging and the v tiles: order before the next TMA and MMA reads
    __syncthreads();
    if (V.abort) break;
    if (n + 1 < nchunks) {
      if (tid == 0) request_z(t0 + kC);
      z_pending = true;
    }
  }

  write_conv_T();
  // After an early exit, no requested copy may still be landing in shared
  // memory, and no MMA still writing TMEM, when the CTA ends: wait (bounded)
  // for any copy that was not consumed and for every MMA issued.
  if (tid == 0) {
    if (raw_pending) bar_wait(&V.bar_raw, phase_raw);
    if (z_pending) bar_wait(&V.bar_z, phase_z);
    for (int j = kq_used; j < kq_next; ++j) bar_wait(&V.bar_kq[j & 1], (uint32_t)(j >> 1) & 1u);
    for (int j = klo_used; j < klo_next; ++j) bar_wait(&V.bar_klo, (uint32_t)j & 1u);
    commit(&V.bar_end);
    bar_wait(&V.bar_end, 0);
  }
  if (issuer2) commit(&V.bar_end);  // the second issuer's MMAs (count 2)
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// A [B][T][width] bf16 tensor as a 3-d map with boxes of 128 columns x `rows` rows.
// The q^ / k^ front end of the staged path, once per key head rather than
// once per value head: conv + SiLU + L2 norm of q and k, written as fp16 q^
// and as an fp16 hi/lo pair for k^ (hi = fp16(k^), lo = fp16(k^ - hi)) into
// qk_ws [3][rows][Hk][128].  The arithmetic is fe_pass's, so q^ and k^'s hi
// part equal the fused kernel's operands bit for bit.
// Persistent: a CTA keeps one key head and takes every nslots-th 64-token
// tile.  A tile's raw q and k rows, with the three before it, arrive by TMA
// in one of kQkStages stages, the next tiles' while this one is computed.
// Half-warps 0-7 take q, 8-15 take k, a run of 8 tokens each, the window
// sliding over the staged rows; a token within three rows of its sequence's
// start takes those rows from the carried window (or zeros) instead.
constexpr int kQkThreads = 256;
constexpr int kQkStages = 2;
constexpr uint32_t kQkStage = 2 * kRawBlock;  // raw q | k rows of one tile
constexpr uint32_t kQkSmem = kQkStages * kQkStage + 64 + 128;  // stages, mbarriers, alignment slack
static_assert(kQkStage % 128 == 0, "TMA stage alignment");

__global__ void __launch_bounds__(kQkThreads, 2)
    prefill_qk_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tm_qkv, int *zero, long long nzero) {
  extern __shared__ uint8_t qk_smem_raw[];
  uint8_t *sm = qk_smem_raw + ((128 - (smem_u32(qk_smem_raw) & 127)) & 127);
  const uint32_t sbase = smem_u32(sm);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + kQkStages * kQkStage);  // a stage's rows landed
  const Dims d = a.d;
  const int kh = (int)(blockIdx.x % (unsigned)d.Hk);
  const int slot = (int)(blockIdx.x / (unsigned)d.Hk), nslots = (int)(gridDim.x / (unsigned)d.Hk);
  const int rows = a.cu_seqlens ? d.T : d.B * d.T;  // token rows fit in 31 bits
  const int ntiles = (rows + kC - 1) / kC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, grp = lane & 15;
  const int hw = 2 * warp + (lane >> 4);  // half-warp 0..15
  const int blk = hw >> 3;                // 0: q, 1: k
  const long long C = d.C;
  const int c = (blk == 0 ? 0 : d.Hk * kD) + kh * kD + 8 * grp;
  const float scale = blk == 0 ? d.q_scale : 1.0f;
  const bf16 *conv_w = static_cast<const bf16 *>(a.conv_w);
  const bf16 *conv0 = static_cast<const bf16 *>(a.conv0);
  for (long long i = (long long)blockIdx.x * kQkThreads + tid; i < nzero; i += (long long)gridDim.x * kQkThreads)
    zero[i] = 0;  // the chunk-parallel prefill's item flags
  if (tid == 0)
    for (int st = 0; st < kQkStages; ++st) bar_init(&full[st], 1);
  __syncthreads();
  // Thread 0: a tile's rows tile*64-3 .. tile*64+63 of this head's q and k
  // channels into a stage (rows outside the tensor read as zeros).
  auto request = [&](int tile, int stage) {
    bar_expect_tx(&full[stage], kQkStage);
    const int row = tile * kC - 3;
    tma_load_3d(sbase + stage * kQkStage, &tm_qkv, kh * kD, row, 0, &full[stage]);
    tma_load_3d(sbase + stage * kQkStage + kRawBlock, &tm_qkv, d.Hk * kD + kh * kD, row, 0, &full[stage]);
  };
  if (tid == 0)
    for (int j = 0; j < kQkStages && slot + j * nslots < ntiles; ++j) request(slot + j * nslots, j);
  float2 w[4][4];  // [channel pair][tap]
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 a0 = ld_io4(conv_w + 4 * (c + 2 * i)), a1 = ld_io4(conv_w + 4 * (c + 2 * i + 1));
    w[i][0] = make_float2(a0.x, a1.x);
    w[i][1] = make_float2(a0.y, a1.y);
    w[i][2] = make_float2(a0.z, a1.z);
    w[i][3] = make_float2(a0.w, a1.w);
  }
  // Outputs: q^ (plane 0), k^ hi and lo (planes 1, 2), row stride Hk * 128.
  const long long rstride = (long long)d.Hk * kD;
  const long long plane = (long long)rows * rstride;
  int n = 0;
  for (int tile = slot; tile < ntiles; tile += nslots, ++n) {
    const int stage = n % kQkStages;
    __syncwarp();
    const bool got = bar_wait(&full[stage], (uint32_t)(n / kQkStages) & 1u);
    if (__syncthreads_or(!got)) {
      if (tid == 0) atomicOr(a.err, kErrTimeout);
      break;
    }
    const int tb = tile * kC + 8 * (hw & 7);  // this half-warp's run: tokens tb .. tb+7
    // this run's window rows tb-3 .. tb+7 in the stage: 256 bytes per row
    const uint8_t *xr = sm + stage * kQkStage + blk * kRawBlock + 256 * (8 * (hw & 7)) + 16 * grp;
    // The sequence of the run's first token, advanced along the run.
    int b = 0, bos = 0, eos = rows;
    if (tb < rows) {
      if (a.cu_seqlens) {  // the last sequence starting at or before tb
        int lo = 0, hi = d.B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (a.cu_seqlens[mid] <= tb) lo = mid; else hi = mid - 1;
        }
        b = lo;
        bos = a.cu_seqlens[b];
        eos = a.cu_seqlens[b + 1];
      } else {
        b = tb / d.T;
        bos = b * d.T;
        eos = bos + d.T;
      }
    }
    __half *dst = static_cast<__half *>(a.qk_ws) + (blk == 0 ? 0 : plane) + (long long)tb * rstride + kh * kD +
                  8 * grp;
    float2 s0[4], s1[4], s2[4];  // the sliding window: rows t-3, t-2, t-1, widened once each
    widen(*reinterpret_cast<const uint4 *>(xr), s0);
    widen(*reinterpret_cast<const uint4 *>(xr + 256), s1);
    widen(*reinterpret_cast<const uint4 *>(xr + 512), s2);
#pragma unroll
    for (int u8 = 0; u8 < 8; ++u8) {
      const int t = tb + u8;
      const bool valid = t < rows;  // the shuffles below run on every lane regardless
      if (valid) {
        while (t >= eos && b + 1 < d.B) {  // the run crossed into the next sequence
          ++b;
          bos = eos;
          eos = a.cu_seqlens ? a.cu_seqlens[b + 1] : bos + d.T;
        }
      }
      float2 x0[4], x1[4], x2[4], x3[4];
      widen(*reinterpret_cast<const uint4 *>(xr + 256 * (u8 + 3)), x3);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x0[i] = s0[i];
        x1[i] = s1[i];
        x2[i] = s2[i];
      }
      if (valid && t - bos < 3) {  // rows before the sequence: the carried window, or zeros
        const bf16 *cw0 = conv0 ? conv0 + (long long)b * 3 * C + c : nullptr;
        const int k0 = t - 3 - bos;  // window row of tap 0: -3 .. -1 -> carried rows 0 .. 2
        const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
        if (k0 < 0) widen(cw0 ? *reinterpret_cast<const uint4 *>(cw0 + (3 + k0) * C) : z4, x0);
        if (k0 + 1 < 0) widen(cw0 ? *reinterpret_cast<const uint4 *>(cw0 + (4 + k0) * C) : z4, x1);
        if (k0 + 2 < 0) widen(cw0 ? *reinterpret_cast<const uint4 *>(cw0 + (5 + k0) * C) : z4, x2);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // slide (the raw rows, not the substituted ones)
        s0[i] = s1[i];
        s1[i] = s2[i];
        s2[i] = x3[i];
      }
      float2 u[4], ss2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 acc = __fmul2_rn(w[i][0], x0[i]);
        acc = __ffma2_rn(w[i][1], x1[i], acc);
        acc = __ffma2_rn(w[i][2], x2[i], acc);
        acc = __ffma2_rn(w[i][3], x3[i], acc);
        u[i] = silu2(acc);
        ss2 = __ffma2_rn(u[i], u[i], ss2);
      }
      float ss = ss2.x + ss2.y;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float f = rsqrtf(ss + d.eps_l2) * scale;
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] = __fmul2_rn(u[i], make_float2(f, f));
      if (valid && in_bounds((dst - static_cast<const __half *>(a.qk_ws)) + (blk == 1 ? plane : 0) + 8, 3 * plane, a.err)) {
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split2_inrange(u[i].x, u[i].y, wh[i], wl[i]);  // |k^|, |q^| <= 1
        *reinterpret_cast<uint4 *>(dst) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        if (blk == 1) *reinterpret_cast<uint4 *>(dst + plane) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
      dst += rstride;
    }
    __syncthreads();  // the stage is read: it may take the tile kQkStages on
    if (tid == 0 && tile + kQkStages * nslots < ntiles) request(tile + kQkStages * nslots, stage);
  }
  // After an early exit no copy may still be landing in shared memory when the
  // CTA ends: wait (bounded) for the requests of the tiles not consumed (on a
  // normal exit there are none).
  if (tid == 0)
    for (int j = n; j < n + kQkStages; ++j)
      if (slot + j * nslots < ntiles) bar_wait(&full[j % kQkStages], (uint32_t)(j / kQkStages) & 1u);
}

// The staged q^ / k^ of qk_ws as a 3-d map {Hk*128 columns, rows, 3 tensors}
// of fp16 with 128-byte-swizzled 64 x 64 boxes: the layout of the K-major
// [K;Q] tile.
bool encode_qk(CUtensorMap *m, void *base, int Hk, long long rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const long long width = (long long)Hk * kD;
  const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)rows, 3};
  const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * rows};
  const cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows(CUtensorMap *m, const void *base, long long width, long long T, int B, int rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * T};
  const cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_chunked(const PrefillArgs &a, bool bf16_io, cudaStream_t s) {
  if (!bf16_io) return cudaErrorInvalidValue;  // the chunked kernel stages bf16 rows
  CUtensorMap tm_qkv, tm_z;
  // The token-major tensors as one run of rows; each CTA addresses its own
  // sequence's rows (fixed length or packed) and masks the rows past its end.
  const long long rows = a.cu_seqlens ? (long long)a.d.T : (long long)a.d.B * a.d.T;
  if (!encode_rows(&tm_qkv, a.qkv_pre, a.d.C, rows, 1, kRawRows) ||
      !encode_rows(&tm_z, a.z, (long long)a.d.Hv * kD, rows, 1, kC))
    return cudaErrorInvalidValue;
  CUtensorMap tm_qk = tm_z;  // unread by the fused variant
  if (a.qk_ws && !encode_qk(&tm_qk, a.qk_ws, a.d.Hk, rows)) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)(a.d.B * a.d.Hv)), block(kThreads);
  const bool raw = a.gate.g == nullptr;
  auto kern = a.qk_ws ? (raw ? prefill_chunked_kernel<true, true> : prefill_chunked_kernel<false, true>)
                      : (raw ? prefill_chunked_kernel<true, false> : prefill_chunked_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, block, kSmemBytes, s>>>(a, tm_qkv, tm_z, tm_qk);
  return cudaGetLastError();
}

cudaError_t launch_prefill_qk(const PrefillArgs &a, cudaStream_t s, int *zero, long long nzero) {
  if (!a.qk_ws) return cudaErrorInvalidValue;
  const long long rows = a.cu_seqlens ? (long long)a.d.T : (long long)a.d.B * a.d.T;
  if (rows <= 0) return cudaSuccess;
  if (rows > 0x7fffffffLL - 2 * kC) return cudaErrorInvalidValue;  // token rows in 31 bits
  CUtensorMap tm_qkv;
  if (!encode_rows(&tm_qkv, a.qkv_pre, a.d.C, rows, 1, kRawRows)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // Two resident CTAs per SM, each keeping one key head.
  const long long ntiles = (rows + kC - 1) / kC;
  long long nslots = (2LL * sms) / a.d.Hk;
  if (nslots > ntiles) nslots = ntiles;
  if (nslots < 1) nslots = 1;
  e = cudaFuncSetAttribute(prefill_qk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQkSmem);
  if (e != cudaSuccess) return e;
  prefill_qk_kernel<<<(unsigned)(nslots * a.d.Hk), kQkThreads, kQkSmem, s>>>(a, tm_qkv, zero, nzero);
  return cudaGetLastError();
}

}  // namespace gdn
