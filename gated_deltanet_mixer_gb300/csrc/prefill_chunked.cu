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
// the 128 value rows as its M dimension:
//   Delta^T = U^T - S W^T        O^T = S (D Q)^T + Delta^T M^T
//   S_out   = d_n S + Delta^T (Gamma K),   M = (Q K^T) o R,  Gamma = diag(d_n / d_j)
// Ratios of decays come from differences of chunk-local cumulative log
// decays G (never a division of two small products); g is clamped at -80.
//
// One CTA per (sequence b, value head h), 8 warps, a sequential loop over the
// chunks.  The fp32 state lives in TMEM for the whole sequence; an fp16 copy
// in shared memory is the MMA operand.  All MMA operands are fp16 (11-bit
// significand; bf16's 8 bits cost several percent of the output's rms at the
// heavy tail of the gated norm) with fp32 accumulation.  The operands that
// feed the state, beta V (through U) and both factors of the state update,
// are carried as hi + lo fp16 pairs (three MMAs for hi*hi + hi*lo + lo*hi),
// which keeps the state within 1e-3 of its rms where single fp16 gives 2e-2
// on short, heavy-tailed updates.  Per chunk, in order:
//   A  conv + SiLU + L2 norms (front end), operand tiles to shared memory
//   B  MMA1  [K;Q] K^T                      -> K K^T, Q K^T
//   C  decayed lower-triangular L (fp32) and M (fp16)
//   D  T = (I + L)^{-1} by forward substitution (fp32, CUDA cores)
//   E  MMA2  U^T = (beta V)^T T^T (hi, lo);  MMA3  W^T = (beta D K)^T T^T
//   F  -W^T to shared memory
//   G  MMA4  Delta^T = U^T - S W^T;  MMA5  O^T = S (D Q)^T
//   H  Delta^T to shared memory
//   I  MMA6  O^T += Delta^T M^T;     MMA7  S += Delta^T (Gamma K) (split)
//   J  gated RMSNorm of O (node gdn.norm) -> o; S -> fp16 copy, rescale for
//      the next chunk (or write S_T after the last)
#include "gdn_device.cuh"
#include "launch.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kC = 64;  // chunk length
constexpr int kThreads = 256;
constexpr float kGMin = -80.0f;

// Shared memory map (byte offsets from a 1024-aligned base).
constexpr uint32_t OFF_KQ = 0;          // [K;Q] K-major, 128 rows x 128     32 KB
constexpr uint32_t OFF_DQ = 32768;      // D Q   K-major,  64 rows x 128     16 KB
constexpr uint32_t OFF_BDK = 49152;     // beta d K  MN-major [j][k]         16 KB
constexpr uint32_t OFF_BV = 65536;      // beta V    MN-major [j][v]         16 KB
constexpr uint32_t OFF_GK = 81920;      // Gamma K   MN-major [j][k]         16 KB
constexpr uint32_t OFF_TM = 98304;      // T         K-major [i][j]           8 KB
constexpr uint32_t OFF_M = 106496;      // M         K-major [i][j]           8 KB
constexpr uint32_t OFF_NW = 114688;     // -W^T      MN-major [k][i]         16 KB
constexpr uint32_t OFF_S = 131072;      // S fp16    K-major [v][k]          32 KB
constexpr uint32_t OFF_DT = 163840;     // Delta^T   K-major [v][j]          16 KB
constexpr uint32_t OFF_GKL = 180224;    // Gamma K, low part                 16 KB
constexpr uint32_t OFF_BVL = 196608;    // beta V, low part                  16 KB
constexpr uint32_t OFF_VEC = 212992;    // per-token vectors and flags        2 KB
constexpr uint32_t OFF_DTL = OFF_KQ;    // Delta^T, low part (aliases [K;Q], dead after MMA1)
constexpr uint32_t OFF_L = OFF_NW;      // L fp32 [64][64] during the solve (aliases -W^T)
constexpr uint32_t OFF_OST = OFF_BDK;   // O^T staging fp32 [64][128] (aliases BDK, BV)
constexpr uint32_t kSmemUsed = OFF_VEC + 2048;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack

// TMEM columns (512 allocated).
constexpr uint32_t TM_S = 0;     // state, fp32 [v][k]          128 columns
constexpr uint32_t TM_O = 128;   // O^T [v][i]                  64
constexpr uint32_t TM_U = 192;   // U^T, then Delta^T [v][j]    64
constexpr uint32_t TM_W = 256;   // W^T [k][i]                  64
constexpr uint32_t TM_KQ = 320;  // [K K^T; Q K^T]              64
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
__device__ __forceinline__ float ratio(const Vecs &V, int i, int j) {
  return V.mild ? V.d[i] * V.dinv[j] : __expf(V.G[i] - V.G[j]);
}

// Chunk vectors from g and beta (one warp).  Padded tokens get g = 0, beta = 0.
__device__ void chunk_vectors(Vecs &V, const float *g, const float *beta, long long gstride,
                              int t0, int T, int lane) {
  float gv[2], bv[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = t0 + lane + 32 * u;
    gv[u] = t < T ? fmaxf(g[(long long)t * gstride], kGMin) : 0.f;
    bv[u] = t < T ? beta[(long long)t * gstride] : 0.f;
  }
  // inclusive scan over 64 = two 32-lane scans
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

template <typename IO>
__device__ __forceinline__ void load8(const IO *p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[8]) {
  uint4 u = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float *p, float (&v)[8]) {
  float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Raw conv input rows: x~[e] for e in [0, T+3): conv0 rows for e < 3, token e-3 after.
template <typename IO>
__device__ __forceinline__ void load_raw8(const IO *x, const IO *conv0, long long C, int t,
                                          int T, long long c, float (&v)[8]) {
  if (t >= 0 && t < T) {
    load8(x + (long long)t * C + c, v);
  } else if (t < 0 && conv0) {
    load8(conv0 + (long long)(3 + t) * C + c, v);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
}

// A: front end for one chunk.  Threads 0..191: quarter (16 tokens) x block
// (q, k, v) x 8-channel group; each slides the conv window over its tokens.
template <typename IO>
__device__ void front_end(uint8_t *sm, const Vecs &V, const PrefillArgs &a, const IO *x,
                          const IO *conv0, int b, int h, int kh, int t0, int tid) {
  if (tid >= 192) return;
  const Dims &d = a.d;
  const long long C = d.C;
  const int quarter = tid / 48, rem = tid % 48, blk = rem / 16, grp = rem % 16;
  const long long c = blk == 0   ? (long long)kh * kD + 8 * grp
                      : blk == 1 ? (long long)d.Hk * kD + (long long)kh * kD + 8 * grp
                                 : 2LL * d.Hk * kD + (long long)h * kD + 8 * grp;
  const IO *cw = static_cast<const IO *>(a.conv_w);
  float w[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 t4 = ld_io4(cw + 4 * (c + i));
    w[i][0] = t4.x; w[i][1] = t4.y; w[i][2] = t4.z; w[i][3] = t4.w;
  }
  const int tb = t0 + 16 * quarter;
  float x0[8], x1[8], x2[8];
  load_raw8(x, conv0, C, tb - 3, d.T, c, x0);
  load_raw8(x, conv0, C, tb - 2, d.T, c, x1);
  load_raw8(x, conv0, C, tb - 1, d.T, c, x2);
  const float scale = blk == 0 ? d.q_scale : 1.0f;
  for (int tt = 0; tt < 16; ++tt) {
    const int t = tb + tt;
    const int row = 16 * quarter + tt;  // token index within the chunk
    float x3[8], u[8];
    load_raw8(x, conv0, C, t, d.T, c, x3);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float acc = w[i][0] * x0[i];
      acc = fmaf(w[i][1], x1[i], acc);
      acc = fmaf(w[i][2], x2[i], acc);
      acc = fmaf(w[i][3], x3[i], acc);
      u[i] = t < d.T ? silu_fast(acc) : 0.f;
      ss = fmaf(u[i], u[i], ss);
      x0[i] = x1[i];
      x1[i] = x2[i];
      x2[i] = x3[i];
    }
    // sum of squares over the 16 groups of this (quarter, block): one half-warp
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (blk < 2) {
      const float f = rsqrtf(ss + d.eps_l2) * scale;
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] *= f;
    }
    float s8[8];
    if (blk == 0) {  // q^: the Q rows of [K;Q], and D Q
      st_h8(sm + OFF_KQ + kmaj(64 + row, 8 * grp, 128), u);
#pragma unroll
      for (int i = 0; i < 8; ++i) s8[i] = u[i] * V.d[row];
      st_h8(sm + OFF_DQ + kmaj(row, 8 * grp, 64), s8);
    } else if (blk == 1) {  // k^: the K rows, beta d K, Gamma K
      st_h8(sm + OFF_KQ + kmaj(row, 8 * grp, 128), u);
#pragma unroll
      for (int i = 0; i < 8; ++i) s8[i] = u[i] * V.bd[row];
      st_h8(sm + OFF_BDK + mnmaj(8 * grp, row, kC), s8);
#pragma unroll
      for (int i = 0; i < 8; ++i) s8[i] = u[i] * V.gam[row];
      st_h8_split(sm + OFF_GK + mnmaj(8 * grp, row, kC), sm + OFF_GKL + mnmaj(8 * grp, row, kC), s8);
    } else {  // v: beta V
#pragma unroll
      for (int i = 0; i < 8; ++i) s8[i] = u[i] * V.beta[row];
      st_h8_split(sm + OFF_BV + mnmaj(8 * grp, row, kC), sm + OFF_BVL + mnmaj(8 * grp, row, kC), s8);
    }
  }
}

// D: T = (I + L)^{-1}, column c by thread c (64 threads), L strictly lower.
// L is fp32 [64][64] with float4 index (j/4) ^ (i % 16) per row.
__device__ void solve_T(uint8_t *sm, int c) {
  const float *L = reinterpret_cast<const float *>(sm + OFF_L);
  float xv[kC];
#pragma unroll
  for (int i = 0; i < kC; ++i) xv[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
  for (int i = 1; i < kC; ++i) {
    float acc = 0.f;
#pragma unroll
    for (int j4 = 0; j4 < i; j4 += 4) {
      const float4 l = reinterpret_cast<const float4 *>(L + i * kC)[(j4 >> 2) ^ (i & 15)];
      acc = fmaf(l.x, xv[j4], acc);
      if (j4 + 1 < i) acc = fmaf(l.y, xv[j4 + 1], acc);
      if (j4 + 2 < i) acc = fmaf(l.z, xv[j4 + 2], acc);
      if (j4 + 3 < i) acc = fmaf(l.w, xv[j4 + 3], acc);
    }
    xv[i] -= acc;
  }
  __half *Tm = reinterpret_cast<__half *>(sm + OFF_TM);
#pragma unroll
  for (int i = 0; i < kC; ++i) Tm[kmaj(i, c, kC) / 2] = to_h(xv[i]);
}

// Issue `nk` K-steps of one MMA family.
struct MmaOp {
  uint32_t d, a_base, b_base, id;
  int a_mode, b_mode;   // 0: K-major, 1: MN-major
  int a_rows, b_rows;   // rows of the K-major tiles
  int a_kdim, b_kdim;   // contraction extent of MN-major tiles
};
__device__ __forceinline__ void issue(const MmaOp &op, int nk, bool accumulate_first) {
  for (int ks = 0; ks < nk; ++ks) {
    const uint64_t ad = op.a_mode ? desc_mn(op.a_base, ks, op.a_kdim) : desc_k(op.a_base, ks, op.a_rows);
    const uint64_t bd = op.b_mode ? desc_mn(op.b_base, ks, op.b_kdim) : desc_k(op.b_base, ks, op.b_rows);
    mma(op.d, ad, bd, op.id, (accumulate_first || ks > 0) ? 1u : 0u);
  }
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
  if (warp == 7) {
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
  {
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
  const uint32_t id_n64_kk = idesc(128, 64, 0, 0);
  const uint32_t id_n64_mk = idesc(128, 64, 1, 0);
  const uint32_t id_n64_km = idesc(128, 64, 0, 1);
  const uint32_t id_n128_km = idesc(128, 128, 0, 1);
  const uint32_t sbase = smem_u32(sm);

  auto mma_sync = [&](bool ok_in) -> bool {
    // all threads: wait for the committed MMAs; uniform abort decision
    bool ok = ok_in && bar_wait(&V.bar, phase);
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
    if (warp == 7) {
      chunk_vectors(V, gp + (long long)t0 * d.Hv, bp + (long long)t0 * d.Hv, d.Hv, 0, T - t0, lane);
      const float dcn = n + 1 < nchunks ? chunk_decay(gp, d.Hv, t0 + kC, T, lane) : 1.f;
      if (lane == 0) V.dC_next = dcn;
    }
    __syncthreads();
    // A: front end
    front_end<IO>(sm, V, a, x, conv0, b, h, kh, t0, tid);
    smem_ready();
    // B: MMA1
    if (tid == 0) {
      fence_after();
      issue(MmaOp{tmem + TM_KQ, sbase + OFF_KQ, sbase + OFF_KQ, id_n64_kk, 0, 0, 128, 128, 0, 0}, 8, false);
      commit(&V.bar);
    }
    if (!mma_sync(true)) break;
    // C: L (fp32, strictly lower, decayed beta K K^T) and M (fp16, decayed Q K^T incl. diagonal)
    {
      float v[32];
      tmem_ld32(tl + TM_KQ + 32 * half, v);
      const int j0 = 32 * half;
      if (lrow < kC) {
        const int i = lrow;
        const float bi = V.beta[i];
        float *L = reinterpret_cast<float *>(sm + OFF_L);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 f;
          const int j = j0 + 4 * q;
          f.x = (j + 0 < i) ? bi * v[4 * q + 0] * ratio(V, i, j + 0) : 0.f;
          f.y = (j + 1 < i) ? bi * v[4 * q + 1] * ratio(V, i, j + 1) : 0.f;
          f.z = (j + 2 < i) ? bi * v[4 * q + 2] * ratio(V, i, j + 2) : 0.f;
          f.w = (j + 3 < i) ? bi * v[4 * q + 3] * ratio(V, i, j + 3) : 0.f;
          reinterpret_cast<float4 *>(L + i * kC)[(j >> 2) ^ (i & 15)] = f;
        }
      } else {
        const int i = lrow - kC;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int j = j0 + q;
          v[q] = (j <= i) ? v[q] * ratio(V, i, j) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) st_h8(sm + OFF_M + kmaj(i, j0 + 8 * q, kC), v + 8 * q);
      }
    }
    __syncthreads();
    // D: the triangular inverse
    if (tid < kC) solve_T(sm, tid);
    smem_ready();
    // E: MMA2, MMA3
    if (tid == 0) {
      fence_after();
      issue(MmaOp{tmem + TM_U, sbase + OFF_BV, sbase + OFF_TM, id_n64_mk, 1, 0, 0, kC, kC, 0}, 4, false);
      issue(MmaOp{tmem + TM_U, sbase + OFF_BVL, sbase + OFF_TM, id_n64_mk, 1, 0, 0, kC, kC, 0}, 4, true);
      issue(MmaOp{tmem + TM_W, sbase + OFF_BDK, sbase + OFF_TM, id_n64_mk, 1, 0, 0, kC, kC, 0}, 4, false);
      commit(&V.bar);
    }
    if (!mma_sync(true)) break;
    // F: -W^T (lanes k, columns i) -> MN-major [k][i]
    {
      float v[32];
      tmem_ld32(tl + TM_W + 32 * half, v);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = -v[q];
#pragma unroll
      for (int q = 0; q < 4; ++q) st_h8(sm + OFF_NW + mnmaj(32 * half + 8 * q, lrow, kD), v + 8 * q);
    }
    smem_ready();
    // G: MMA4 (Delta^T = U^T - S W^T), MMA5 (O^T = S (D Q)^T)
    if (tid == 0) {
      fence_after();
      issue(MmaOp{tmem + TM_U, sbase + OFF_S, sbase + OFF_NW, id_n64_km, 0, 1, 128, 0, 0, kD}, 8, true);
      issue(MmaOp{tmem + TM_O, sbase + OFF_S, sbase + OFF_DQ, id_n64_kk, 0, 0, 128, kC, 0, 0}, 8, false);
      commit(&V.bar);
    }
    if (!mma_sync(true)) break;
    // H: Delta^T (lanes v, columns j) -> K-major [v][j]
    {
      float v[32];
      tmem_ld32(tl + TM_U + 32 * half, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t o = kmaj(lrow, 32 * half + 8 * q, 128);
        st_h8_split(sm + OFF_DT + o, sm + OFF_DTL + o, v + 8 * q);
      }
    }
    smem_ready();
    // I: MMA6 (O^T += Delta^T M^T), MMA7 (S += Delta^T Gamma K)
    if (tid == 0) {
      fence_after();
      issue(MmaOp{tmem + TM_O, sbase + OFF_DT, sbase + OFF_M, id_n64_kk, 0, 0, 128, kC, 0, 0}, 4, true);
      issue(MmaOp{tmem + TM_S, sbase + OFF_DT, sbase + OFF_GK, id_n128_km, 0, 1, 128, 0, 0, kC}, 4, true);
      issue(MmaOp{tmem + TM_S, sbase + OFF_DT, sbase + OFF_GKL, id_n128_km, 0, 1, 128, 0, 0, kC}, 4, true);
      issue(MmaOp{tmem + TM_S, sbase + OFF_DTL, sbase + OFF_GK, id_n128_km, 0, 1, 128, 0, 0, kC}, 4, true);
      commit(&V.bar);
    }
    if (!mma_sync(true)) break;
    // J1: O^T -> staging [i][v]; S -> fp16 copy and rescaled TMEM state (or S_T)
    {
      float *ost = reinterpret_cast<float *>(sm + OFF_OST);
      float v[32];
      tmem_ld32(tl + TM_O + 32 * half, v);
#pragma unroll
      for (int q = 0; q < 32; ++q) ost[(32 * half + q) * kD + lrow] = v[q];
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
    // J2: gated RMSNorm per token, one warp per token
    {
      const float *ost = reinterpret_cast<const float *>(sm + OFF_OST);
      const float4 w4 = ld_io4(static_cast<const IO *>(a.norm_w) + 4 * lane);
      const int nv = min(kC, T - t0);
      for (int i = warp; i < nv; i += 8) {
        const float4 o4 = reinterpret_cast<const float4 *>(ost + i * kD)[lane];
        const float rstd = rsqrtf(warp_sum(dot4(o4, o4)) * (1.0f / kD) + d.eps_norm);
        const long long oi = (((long long)b * T + t0 + i) * d.Hv + h) * kD + 4 * lane;
        const float4 z4 = ld_io4(static_cast<const IO *>(a.z) + oi);
        float4 y;
        y.x = w4.x * (o4.x * rstd) * silu_fast(z4.x);
        y.y = w4.y * (o4.y * rstd) * silu_fast(z4.y);
        y.z = w4.z * (o4.z * rstd) * silu_fast(z4.z);
        y.w = w4.w * (o4.w * rstd) * silu_fast(z4.w);
        st_io4(static_cast<IO *>(a.o) + oi, y);
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
