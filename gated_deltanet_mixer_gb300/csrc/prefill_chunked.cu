// prefill_chunked.cu -- the chunked (WY) form of the gated delta rule on the
// tcgen05 tensor cores.
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
// chunks.  The fp32 state lives in TMEM for the whole sequence; an fp16 copy
// in shared memory is the MMA operand.  All MMA operands are fp16 (11-bit
// significand; bf16's 8 bits cost several percent of the output's rms at the
// heavy tail of the gated norm) with fp32 accumulation.  The operands that
// feed the state, V and T B (through U) and both factors of the state update,
// are carried as hi + lo fp16 pairs (three MMAs for hi*hi + hi*lo + lo*hi), which
// keeps the state within about 1e-3 of its rms where single fp16 gives 2e-2
// on short, heavy-tailed updates.  Per chunk, in order:
//   A  conv + SiLU + L2 norms (front end), operand tiles to shared memory
//   B  MMA1  [K;Q] K^T                        -> K K^T, Q K^T
//   C  decayed lower-triangular L (fp32) and M (fp16)
//   D  T = (I + L)^{-1} in 16 x 16 blocks (fp32, CUDA cores) -> T B, T B D
//   E  MMA2  U^T = V^T (T B)^T (split);  MMA3  W^T = K^T (T B D)^T
//   F  -W^T to shared memory
//   G  MMA4  Delta^T = U^T - S W^T;  MMA5  S Q^T
//   H  Delta^T (hi, lo) to shared memory
//   I  MMA6  Delta^T M^T;            MMA7  S += Delta^T (Gamma K) (split)
//   J  O = d (S Q^T) + Delta^T M^T, gated RMSNorm (node gdn.norm) -> o;
//      S -> fp16 copy, rescaled for the next chunk (or S_T after the last)
#include "gdn_device.cuh"
#include "launch.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kC = 64;  // chunk length
constexpr int kThreads = 384;   // 12 warps
constexpr int kTmemWarps = 8;   // warps 0..7 do the TMEM <-> register passes (two per lane quadrant)
constexpr float kGMin = -80.0f;

// Shared memory map (byte offsets from a 1024-aligned base).  fp16 tiles.
constexpr uint32_t OFF_KQ = 0;          // [K;Q] K-major, 128 rows x 128       32 KB
constexpr uint32_t OFF_VH = 32768;      // V hi      MN-major [j][v]           16 KB
constexpr uint32_t OFF_VL = 49152;      // V lo                                16 KB
constexpr uint32_t OFF_GK = 65536;      // Gamma K hi  MN-major [j][k]         16 KB
constexpr uint32_t OFF_GKL = 81920;     // Gamma K lo                          16 KB
constexpr uint32_t OFF_TU = 98304;      // T diag(beta)      K-major [i][j]     8 KB
constexpr uint32_t OFF_TW = 106496;     // T diag(beta d)    K-major [i][j]     8 KB
constexpr uint32_t OFF_M = 114688;      // M         K-major [i][j]             8 KB
constexpr uint32_t OFF_NW = 122880;     // -W^T      MN-major [k][i]           16 KB
constexpr uint32_t OFF_S = 139264;      // S         K-major [v][k]            32 KB
constexpr uint32_t OFF_DT = 172032;     // Delta^T hi K-major [v][j]           16 KB
constexpr uint32_t OFF_DTL = 188416;    // Delta^T lo                          16 KB
constexpr uint32_t OFF_TUL = 204800;    // T diag(beta), low part               8 KB
constexpr uint32_t OFF_VEC = 212992;    // per-token vectors and flags          2 KB
// Scratch that lives only between two uses of the tiles it overlays:
constexpr int kLs = 68;                 // padded row stride of L (floats)
constexpr uint32_t OFF_L = OFF_DT;      // L fp32 [64][68], phases C-D (DT and the start of DTL)
constexpr uint32_t OFF_PB = OFF_DT + 64 * kLs * 4;  // block products fp32 [3][16][16], phase D
constexpr uint32_t OFF_TF = OFF_NW;     // T fp32 [64][64], phase D
constexpr uint32_t OFF_OST = OFF_VH;    // O^T staging fp32 [64][128] (VH + VL), phase J
constexpr uint32_t kSmemUsed = OFF_VEC + 2048;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack

// TMEM columns (512 allocated).
constexpr uint32_t TM_S = 0;      // state, fp32 [v][k]           128 columns
constexpr uint32_t TM_O1 = 128;   // S Q^T [v][i]                 64
constexpr uint32_t TM_O2 = 192;   // Delta^T M^T [v][i]           64
constexpr uint32_t TM_U = 256;    // U^T, then Delta^T [v][j]     64
constexpr uint32_t TM_W = 320;    // W^T [k][i]                   64
constexpr uint32_t TM_KQ = 384;   // [K K^T; Q K^T]               64
constexpr uint32_t kTmemCols = 512;

struct Vecs {  // per-token chunk vectors in shared memory
  float G[kC];     // chunk-local cumulative log decay
  float d[kC];     // e^{G_i}
  float dinv[kC];  // e^{-G_j} (only when the chunk's decay is mild)
  float gam[kC];   // e^{G_last - G_j}
  float beta[kC];
  float bd[kC];    // beta_j d_j
  float dC;        // e^{G_last} of the current chunk
  float dC_next;   // e^{G_last} of the next chunk
  int mild;        // G_last >= -40: ratios as d_i * dinv_j
  int abort;
  uint32_t tmem;
  uint64_t bar;
};
static_assert(sizeof(Vecs) <= 2048, "vector area");

__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// e^{G_i - G_j} for j <= i
__device__ __forceinline__ float ratio(const Vecs &V, bool mild, int i, int j) {
  return mild ? V.d[i] * V.dinv[j] : __expf(V.G[i] - V.G[j]);
}

// Chunk vectors from g and beta (one warp).  Padded tokens get g = 0, beta = 0.
__device__ void chunk_vectors(Vecs &V, const float *g, const float *beta, long long gstride,
                              int T, int lane) {
  float gv[2], bv[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = lane + 32 * u;
    gv[u] = t < T ? fmaxf(g[(long long)t * gstride], kGMin) : 0.f;
    bv[u] = t < T ? beta[(long long)t * gstride] : 0.f;
  }
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
  if (lane == 0) {
    V.dC = __expf(Glast);
    V.mild = mild ? 1 : 0;
  }
}

// e^{sum of the chunk's clamped g} for the chunk starting at t0 (one warp).
__device__ float chunk_decay(const float *g, long long gstride, int t0, int T, int lane) {
  float s = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = t0 + lane + 32 * u;
    s += t < T ? fmaxf(g[(long long)t * gstride], kGMin) : 0.f;
  }
  return __expf(warp_sum(s));
}

// Eight consecutive raw io values of one row, as loaded (not yet widened).
template <typename IO>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 u;
};
template <>
struct Raw8<float> {
  float4 a, b;
};

// Raw conv input x~[t] (token t; t < 0 reads the carried window, t >= T reads 0).
template <typename IO>
__device__ __forceinline__ Raw8<IO> ld_raw8(const IO *x, const IO *conv0, long long C, int t,
                                            int T, long long c) {
  Raw8<IO> r;
  const IO *p = nullptr;
  if (t >= 0 && t < T) p = x + (long long)t * C + c;
  else if (t < 0 && conv0) p = conv0 + (long long)(3 + t) * C + c;
  if constexpr (sizeof(IO) == 2) {
    r.u = p ? *reinterpret_cast<const uint4 *>(p) : make_uint4(0, 0, 0, 0);
  } else {
    r.a = p ? reinterpret_cast<const float4 *>(p)[0] : make_float4(0.f, 0.f, 0.f, 0.f);
    r.b = p ? reinterpret_cast<const float4 *>(p)[1] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  return r;
}
// Widen to four channel pairs.
__device__ __forceinline__ void widen(const Raw8<__nv_bfloat16> &r, float2 (&v)[4]) {
  const uint32_t w[4] = {r.u.x, r.u.y, r.u.z, r.u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
__device__ __forceinline__ void widen(const Raw8<float> &r, float2 (&v)[4]) {
  v[0] = make_float2(r.a.x, r.a.y);
  v[1] = make_float2(r.a.z, r.a.w);
  v[2] = make_float2(r.b.x, r.b.y);
  v[3] = make_float2(r.b.z, r.b.w);
}

// 16 bytes of fp16 (8 values, packed conversions, no range clamp: the caller
// guarantees finite fp16 range) to shared memory.
__device__ __forceinline__ void st_h8_fast(uint8_t *p, const float *v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 t = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&t);
  }
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// A: front end for one chunk.  All 12 warps: warp w handles block w / 4
// (q, k, v), two 8-token eighths (one per half-warp) and, per lane, one
// 8-channel group; each thread slides the conv window over its 8 tokens, four
// at a time, with the next four rows already in flight.  Every warp runs the
// same code; what differs per block (norm, outputs) is warp-uniform data.
// Writes: q^ and k^ (fp16) into [K;Q]; Gamma k^ (hi, lo); v (hi, lo).
template <typename IO>
__device__ void front_end(uint8_t *sm, const Vecs &V, const PrefillArgs &a, const IO *x,
                          const IO *conv0, int h, int kh, int t0, int tid) {
  const Dims &d = a.d;
  const long long C = d.C;
  const int warp = tid >> 5, lane = tid & 31;
  const int blk = warp >> 2, eighth = 2 * (warp & 3) + (lane >> 4), grp = lane & 15;
  const long long c = blk == 0   ? (long long)kh * kD + 8 * grp
                      : blk == 1 ? (long long)d.Hk * kD + (long long)kh * kD + 8 * grp
                                 : 2LL * d.Hk * kD + (long long)h * kD + 8 * grp;
  // warp-uniform output plan
  const bool has_norm = blk < 2, has_single = blk < 2, has_split = blk > 0, has_gamma = blk == 1;
  const int row_off = blk == 0 ? 64 : 0;
  const float scale = blk == 0 ? d.q_scale : 1.0f;
  uint8_t *const dhi = sm + (blk == 1 ? OFF_GK : OFF_VH);
  uint8_t *const dlo = sm + (blk == 1 ? OFF_GKL : OFF_VL);
  const IO *cw = static_cast<const IO *>(a.conv_w);
  float2 w[4][4];  // [channel pair][tap]
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 a0 = ld_io4(cw + 4 * (c + 2 * i)), a1 = ld_io4(cw + 4 * (c + 2 * i + 1));
    w[i][0] = make_float2(a0.x, a1.x);
    w[i][1] = make_float2(a0.y, a1.y);
    w[i][2] = make_float2(a0.z, a1.z);
    w[i][3] = make_float2(a0.w, a1.w);
  }
  const int tb = t0 + 8 * eighth;
  float2 x0[4], x1[4], x2[4];
  {
    const Raw8<IO> h0 = ld_raw8(x, conv0, C, tb - 3, d.T, c), h1 = ld_raw8(x, conv0, C, tb - 2, d.T, c),
                   h2 = ld_raw8(x, conv0, C, tb - 1, d.T, c);
    widen(h0, x0);
    widen(h1, x1);
    widen(h2, x2);
  }
  Raw8<IO> nx[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) nx[e] = ld_raw8(x, conv0, C, tb + e, d.T, c);

  auto token = [&](const Raw8<IO> &raw, int tt) {
    const int t = tb + tt;
    const int row = 8 * eighth + tt;  // token index within the chunk
    float2 x3[4];
    widen(raw, x3);
    float u[8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 acc = __fmul2_rn(w[i][0], x0[i]);
      acc = __ffma2_rn(w[i][1], x1[i], acc);
      acc = __ffma2_rn(w[i][2], x2[i], acc);
      acc = __ffma2_rn(w[i][3], x3[i], acc);
      u[2 * i] = t < d.T ? silu_fast(acc.x) : 0.f;
      u[2 * i + 1] = t < d.T ? silu_fast(acc.y) : 0.f;
      ss = fmaf(u[2 * i], u[2 * i], fmaf(u[2 * i + 1], u[2 * i + 1], ss));
      x0[i] = x1[i];
      x1[i] = x2[i];
      x2[i] = x3[i];
    }
    // sum of squares over the 16 groups of this eighth: one half-warp
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float f = has_norm ? rsqrtf(ss + d.eps_l2) * scale : 1.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] *= f;
    if (has_single) st_h8_fast(sm + OFF_KQ + kmaj(row_off + row, 8 * grp, 128), u);
    if (has_split) {
      const float gm = has_gamma ? V.gam[row] : 1.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] *= gm;
      const uint32_t o = mnmaj(8 * grp, row, kC);
      st_h8_split(dhi + o, dlo + o, u);
    }
  };

#pragma unroll 1
  for (int g4 = 0; g4 < 8; g4 += 4) {
    Raw8<IO> cur[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) cur[e] = nx[e];
    if (g4 + 4 < 8) {
#pragma unroll
      for (int e = 0; e < 4; ++e) nx[e] = ld_raw8(x, conv0, C, tb + g4 + 4 + e, d.T, c);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) token(cur[e], g4 + e);
  }
}

// D: T = (I + L)^{-1} in 16 x 16 blocks (all threads).  The diagonal blocks
// by forward substitution, one column per thread; then, block row by block
// row, T_IJ = -T_II sum_{K=J}^{I-1} L_IK T_KJ.  fp32 throughout; the result is
// written as the fp16 K-major tiles T diag(beta) (hi, lo) and T diag(beta d).
// L is [64][kLs] (padded rows), T is [64][64].
__device__ void solve_T(uint8_t *sm, const Vecs &V, int tid) {
  const float *L = reinterpret_cast<const float *>(sm + OFF_L);
  float *Tf = reinterpret_cast<float *>(sm + OFF_TF);
  float *P = reinterpret_cast<float *>(sm + OFF_PB);
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
      for (int j = 0; j < i; ++j) {
        if (j & 1) a1 = fmaf(Lb[i * kLs + j], xv[j], a1);
        else a0 = fmaf(Lb[i * kLs + j], xv[j], a0);
      }
      xv[i] -= a0 + a1;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tf[(base + i) * kC + base + c] = xv[i];
  }
  __syncthreads();
  const bool worker = tid < 256;
  const int r = (tid >> 4) & 15, c = tid & 15;
#pragma unroll 1
  for (int I = 1; I < 4; ++I) {
    const float *Lr = L + (16 * I + r) * kLs;
#pragma unroll 1
    for (int J = 0; J < (worker ? I : 0); ++J) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll 1
      for (int K = J; K < I; ++K) {
        const float *l = Lr + 16 * K;
        const float *t = Tf + 16 * K * kC + 16 * J + c;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          a0 = fmaf(l[k], t[k * kC], a0);
          a1 = fmaf(l[k + 1], t[(k + 1) * kC], a1);
        }
      }
      P[J * 256 + r * 16 + c] = a0 + a1;
    }
    __syncthreads();
    const float *Tii = Tf + (16 * I + r) * kC + 16 * I;
#pragma unroll 1
    for (int J = 0; J < (worker ? I : 0); ++J) {
      const float *pj = P + J * 256 + c;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int k = 0; k < 16; k += 2) {
        s0 = fmaf(Tii[k], pj[k * 16], s0);
        s1 = fmaf(Tii[k + 1], pj[(k + 1) * 16], s1);
      }
      Tf[(16 * I + r) * kC + 16 * J + c] = -(s0 + s1);
    }
    __syncthreads();
  }
  // fp16 tiles: 512 chunks of 8 each, two per thread; blocks above the diagonal are zero
#pragma unroll 1
  for (int m = 0; m < (worker ? 2 : 0); ++m) {
    const int q = tid + 256 * m, i = q >> 3, j0 = (q & 7) * 8;
    const bool below = (j0 >> 4) <= (i >> 4);
    float tb[8], tw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float t = below ? Tf[i * kC + j0 + u] : 0.f;
      tb[u] = t * V.beta[j0 + u];
      tw[u] = t * V.bd[j0 + u];
    }
    st_h8_split(sm + OFF_TU + kmaj(i, j0, kC), sm + OFF_TUL + kmaj(i, j0, kC), tb);
    st_h8(sm + OFF_TW + kmaj(i, j0, kC), tw);
  }
}

// K steps of one MMA family; descriptors built by the caller's lambdas.
template <typename FA, typename FB>
__device__ __forceinline__ void issue(uint32_t d, uint32_t id, int nk, bool accumulate_first, FA da, FB db) {
  for (int ks = 0; ks < nk; ++ks) mma(d, da(ks), db(ks), id, (accumulate_first || ks > 0) ? 1u : 0u);
}

template <typename IO>
__global__ void __launch_bounds__(kThreads, 1) prefill_chunked_kernel(PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Vecs &V = *reinterpret_cast<Vecs *>(sm + OFF_VEC);
  const Dims d = a.d;
  const int unit = blockIdx.x;
  const int b = unit / d.Hv, h = unit % d.Hv;
  const int r = d.Hv / d.Hk, kh = h / r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = d.T;
  const long long C = d.C;
  const IO *x = static_cast<const IO *>(a.qkv_pre) + (long long)b * T * C;
  const IO *conv0 = a.conv0 ? static_cast<const IO *>(a.conv0) + (long long)b * 3 * C : nullptr;
  const float *gp = a.g + (long long)b * T * d.Hv + h;
  const float *bp = a.beta + (long long)b * T * d.Hv + h;
  const long long unit_off = ((long long)b * d.Hv + h) * kD * kD;

  if (tid == 0) {
    bar_init(&V.bar, 1);
    V.abort = 0;
  }
  if (warp == 0) tmem_alloc(&V.tmem, kTmemCols);
  if (warp == 11) {
    const float dc0 = chunk_decay(gp, d.Hv, 0, T, lane);
    if (lane == 0) V.dC_next = dc0;
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = V.tmem;
  // TMEM lane quadrant and column half of this warp for the 32x32b accesses.
  const int quad = warp & 3, half = warp >> 2;
  const int lrow = 32 * quad + lane;  // TMEM lane (row) this thread reads
  const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);

  // Initial state: TMEM <- dC(chunk 0) * S0, shared fp16 copy <- S0.
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
#pragma unroll
      for (int q = 0; q < 4; ++q) st_h8(sm + OFF_S + kmaj(lrow, k0 + 8 * q, 128), v + 8 * q);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] *= dc0;
      tmem_st32(tl + TM_S + k0, v);
    }
  }

  uint32_t phase = 0;
  const int nchunks = (T + kC - 1) / kC;
  const uint32_t id_kk = idesc(128, 64, 0, 0);
  const uint32_t id_mk = idesc(128, 64, 1, 0);
  const uint32_t id_km = idesc(128, 64, 0, 1);
  const uint32_t id_km128 = idesc(128, 128, 0, 1);
  const uint32_t sbase = smem_u32(sm);

  auto mma_sync = [&]() -> bool {
    // all threads: wait for the committed MMAs; uniform abort decision
    bool ok = bar_wait(&V.bar, phase);
    phase ^= 1u;
    fence_after();
    const int bad = __syncthreads_or(!ok);
    if (bad && tid == 0) {
      atomicOr(a.err, kErrTimeout);
      V.abort = 1;
    }
    return !bad;
  };
  auto smem_ready = [&]() {  // shared-memory operands written -> visible to the MMA unit
    fence_smem_to_async();
    fence_before();
    __syncthreads();
  };

  for (int n = 0; n < nchunks; ++n) {
    const int t0 = n * kC;
    // A0: chunk vectors; the next chunk's total decay
    if (warp == 11) {
      chunk_vectors(V, gp + (long long)t0 * d.Hv, bp + (long long)t0 * d.Hv, d.Hv, T - t0, lane);
      const float dcn = n + 1 < nchunks ? chunk_decay(gp, d.Hv, t0 + kC, T, lane) : 1.f;
      if (lane == 0) V.dC_next = dcn;
    }
    __syncthreads();
    // A: front end
    front_end<IO>(sm, V, a, x, conv0, h, kh, t0, tid);
    smem_ready();
    // B: MMA1  [K;Q] K^T
    if (tid == 0) {
      fence_after();
      issue(tmem + TM_KQ, id_kk, 8, false, [&](int ks) { return desc_k(sbase + OFF_KQ, ks, 128); },
            [&](int ks) { return desc_k(sbase + OFF_KQ, ks, 128); });
      commit(&V.bar);
    }
    if (!mma_sync()) break;
    // C: L (fp32, strictly lower, decayed beta K K^T) and M (fp16, decayed Q K^T incl. diagonal)
    if (warp < kTmemWarps) {
      float v[32];
      tmem_ld32(tl + TM_KQ + 32 * half, v);
      const int j0 = 32 * half;
      const bool mild = V.mild != 0;
      if (lrow < kC) {
        const int i = lrow;
        const float bi = V.beta[i];
        float *L = reinterpret_cast<float *>(sm + OFF_L);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 f;
          const int j = j0 + 4 * q;
          f.x = (j + 0 < i) ? bi * v[4 * q + 0] * ratio(V, mild, i, j + 0) : 0.f;
          f.y = (j + 1 < i) ? bi * v[4 * q + 1] * ratio(V, mild, i, j + 1) : 0.f;
          f.z = (j + 2 < i) ? bi * v[4 * q + 2] * ratio(V, mild, i, j + 2) : 0.f;
          f.w = (j + 3 < i) ? bi * v[4 * q + 3] * ratio(V, mild, i, j + 3) : 0.f;
          *reinterpret_cast<float4 *>(L + i * kLs + j) = f;
        }
      } else {
        const int i = lrow - kC;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int j = j0 + q;
          v[q] = (j <= i) ? v[q] * ratio(V, mild, i, j) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) st_h8(sm + OFF_M + kmaj(i, j0 + 8 * q, kC), v + 8 * q);
      }
    }
    __syncthreads();
    // D: the triangular inverse, scaled copies T B and T B D
    solve_T(sm, V, tid);
    smem_ready();
    // E: MMA2 U^T = V^T (T B)^T, hi*hi + lo*hi + hi*lo; MMA3 W^T = K^T (T B D)^T
    // (K^ read from [K;Q] as an MN-major operand)
    if (tid == 0) {
      fence_after();
      auto a_vh = [&](int ks) { return desc_mn(sbase + OFF_VH, ks, kC); };
      auto b_tu = [&](int ks) { return desc_k(sbase + OFF_TU, ks, kC); };
      issue(tmem + TM_U, id_mk, 4, false, a_vh, b_tu);
      issue(tmem + TM_U, id_mk, 4, true, [&](int ks) { return desc_mn(sbase + OFF_VL, ks, kC); }, b_tu);
      issue(tmem + TM_U, id_mk, 4, true, a_vh, [&](int ks) { return desc_k(sbase + OFF_TUL, ks, kC); });
      issue(tmem + TM_W, id_mk, 4, false,
            [&](int ks) { return desc(sbase + OFF_KQ + (uint32_t)(ks * 2048), 128 * 128, 1024); },
            [&](int ks) { return desc_k(sbase + OFF_TW, ks, kC); });
      commit(&V.bar);
    }
    if (!mma_sync()) break;
    // F: -W^T (lanes k, columns i) -> MN-major [k][i]
    if (warp < kTmemWarps) {
      float v[32];
      tmem_ld32(tl + TM_W + 32 * half, v);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = -v[q];
#pragma unroll
      for (int q = 0; q < 4; ++q) st_h8(sm + OFF_NW + mnmaj(32 * half + 8 * q, lrow, kD), v + 8 * q);
    }
    smem_ready();
    // G: MMA4 Delta^T = U^T - S W^T;  MMA5 S Q^T (Q^ = rows 64..127 of [K;Q])
    if (tid == 0) {
      fence_after();
      auto a_s = [&](int ks) { return desc_k(sbase + OFF_S, ks, 128); };
      issue(tmem + TM_U, id_km, 8, true, a_s, [&](int ks) { return desc_mn(sbase + OFF_NW, ks, kD); });
      issue(tmem + TM_O1, id_kk, 8, false, a_s, [&](int ks) { return desc_k(sbase + OFF_KQ + 64 * 128, ks, 128); });
      commit(&V.bar);
    }
    if (!mma_sync()) break;
    // H: Delta^T (lanes v, columns j) -> K-major [v][j], hi and lo
    if (warp < kTmemWarps) {
      float v[32];
      tmem_ld32(tl + TM_U + 32 * half, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t o = kmaj(lrow, 32 * half + 8 * q, 128);
        st_h8_split(sm + OFF_DT + o, sm + OFF_DTL + o, v + 8 * q);
      }
    }
    smem_ready();
    // I: MMA6 Delta^T M^T;  MMA7 S += Delta^T (Gamma K), hi*hi + hi*lo + lo*hi
    if (tid == 0) {
      fence_after();
      auto a_dt = [&](int ks) { return desc_k(sbase + OFF_DT, ks, 128); };
      auto b_gk = [&](int ks) { return desc_mn(sbase + OFF_GK, ks, kC); };
      issue(tmem + TM_O2, id_kk, 4, false, a_dt, [&](int ks) { return desc_k(sbase + OFF_M, ks, kC); });
      issue(tmem + TM_S, id_km128, 4, true, a_dt, b_gk);
      issue(tmem + TM_S, id_km128, 4, true, a_dt, [&](int ks) { return desc_mn(sbase + OFF_GKL, ks, kC); });
      issue(tmem + TM_S, id_km128, 4, true, [&](int ks) { return desc_k(sbase + OFF_DTL, ks, 128); }, b_gk);
      commit(&V.bar);
    }
    if (!mma_sync()) break;
    // J1: O^T = d (S Q^T) + Delta^T M^T -> staging [i][v]; S -> fp16 copy and
    // rescaled TMEM state (or S_T after the last chunk)
    if (warp < kTmemWarps) {
      float *ost = reinterpret_cast<float *>(sm + OFF_OST);
      float v[32], w2[32];
      tmem_ld32(tl + TM_O1 + 32 * half, v);
      tmem_ld32(tl + TM_O2 + 32 * half, w2);
#pragma unroll
      for (int q = 0; q < 32; ++q) ost[(32 * half + q) * kD + lrow] = fmaf(V.d[32 * half + q], v[q], w2[q]);
      const bool last = n + 1 == nchunks;
      const float dcn = V.dC_next;
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int k0 = 64 * half + 32 * p;
        tmem_ld32(tl + TM_S + k0, v);
        if (last) {
          float4 *dst = reinterpret_cast<float4 *>(a.S_T + unit_off + (long long)lrow * kD + k0);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) st_h8(sm + OFF_S + kmaj(lrow, k0 + 8 * q, 128), v + 8 * q);
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] *= dcn;
          tmem_st32(tl + TM_S + k0, v);
        }
      }
    }
    fence_before();
    __syncthreads();
    // J2: gated RMSNorm per token, one warp per token (z rows loaded first)
    {
      const float *ost = reinterpret_cast<const float *>(sm + OFF_OST);
      const float4 w4 = ld_io4(static_cast<const IO *>(a.norm_w) + 4 * lane);
      const int nv = min(kC, T - t0);
      const IO *zb = static_cast<const IO *>(a.z) + (((long long)b * T + t0) * d.Hv + h) * kD + 4 * lane;
      const long long zstride = (long long)d.Hv * kD;
      constexpr int kNW = kThreads / 32, kPer = (kC + kNW - 1) / kNW;
      float4 z4[kPer];
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int i = warp + kNW * m;
        z4[m] = i < nv ? ld_io4(zb + i * zstride) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      IO *ob = static_cast<IO *>(a.o) + (((long long)b * T + t0) * d.Hv + h) * kD + 4 * lane;
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int i = warp + kNW * m;
        if (i < nv) {
          const float4 o4 = reinterpret_cast<const float4 *>(ost + i * kD)[lane];
          const float rstd = rsqrtf(warp_sum(dot4(o4, o4)) * (1.0f / kD) + d.eps_norm);
          float4 y;
          y.x = w4.x * (o4.x * rstd) * silu_fast(z4[m].x);
          y.y = w4.y * (o4.y * rstd) * silu_fast(z4[m].y);
          y.z = w4.z * (o4.z * rstd) * silu_fast(z4[m].z);
          y.w = w4.w * (o4.w * rstd) * silu_fast(z4[m].w);
          st_io4(ob + i * zstride, y);
        }
      }
    }
    __syncthreads();
  }

  // Carried conv window: the last three raw rows of the channels this CTA owns.
  {
    IO *cT = static_cast<IO *>(a.conv_T) + (long long)b * 3 * C;
    const bool own_qk = (h % r) == 0;
    for (int idx = tid; idx < 3 * 3 * kD; idx += kThreads) {
      const int e = idx / (3 * kD), rem = idx % (3 * kD), blk = rem / kD, ch = rem % kD;
      if (blk < 2 && !own_qk) continue;
      const long long c = blk == 0   ? (long long)kh * kD + ch
                          : blk == 1 ? (long long)d.Hk * kD + (long long)kh * kD + ch
                                     : 2LL * d.Hk * kD + (long long)h * kD + ch;
      const int t = T - 3 + e;
      IO val;
      if (t >= 0) val = x[(long long)t * C + c];
      else if (conv0) val = conv0[(long long)(3 + t) * C + c];
      else val = IO(0.f);
      cT[(long long)e * C + c] = val;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill_chunked(const PrefillArgs &a, bool bf16, cudaStream_t s) {
  dim3 grid((unsigned)(a.d.B * a.d.Hv)), block(kThreads);
  cudaError_t e;
  if (bf16) {
    e = cudaFuncSetAttribute(prefill_chunked_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_chunked_kernel<__nv_bfloat16><<<grid, block, kSmemBytes, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(prefill_chunked_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_chunked_kernel<float><<<grid, block, kSmemBytes, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
