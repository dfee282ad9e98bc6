// prefill_split.cu -- the chunked (WY) prefill split into a chunk-parallel
// part and a sequential part, so that only the state recurrence is serial.
//
// Page "How Qwen3.5 works" (azmle112.github.io), section 9.11: within a chunk
// of 64 tokens, A = I + tril((B K K^T) o R, -1), T = A^{-1}, U = T B V and
// W = T B D K depend on the chunk alone; only Delta = U - W S, the output
// O = D Q S + ((Q K^T) o R) Delta and the state update
// S <- d_n S + K^T diag(d_n / d_j) Delta need the carried state S.  Kept
// value-major (S[v][k], node gdn.core of the Qwen3.8-27B spec):
//   Delta^T = U^T - S W^T,  O^T = (S Q^T) D + Delta^T M^T,  M = (Q K^T) o R,
//   S <- d_n S + (Delta Gamma)^T K,  Gamma = diag(d_n / d_j).
//
// prefill_prep_kernel, one work item per (chunk, value head), every chunk of
// every sequence at once (persistent CTAs, two per SM): from the staged q^ and
// k^ of the chunk (written once per key head by prefill_qk_kernel) and its raw
// v rows and gates it forms the chunk vectors, [K;Q] K^T on the tensor cores,
// L and M, the inverse T (fp32, CUDA cores), the v tiles (conv + SiLU, into
// TMEM as fp16 hi/lo), U^T = V^T (T B)^T and -W^T = K^T (-T B D)^T on the
// tensor cores, and writes U^T (fp32), -W^T (fp16), M (fp16) and the vectors
// d, Gamma to a workspace.
//
// prefill_seq_kernel, one CTA per (sequence, value head): walks the chunks
// with the fp32 state resident in TMEM.  Per chunk four groups of MMAs:
//   MMA4  D = S (-W^T)        MMA5  O1 = S Q^T
//   MMA6  O2 = Delta^T M^T    MMA7  S += (Delta Gamma)^T K (hi/lo split)
// and three passes on the CUDA cores: Delta = D + U^T to fp16 (hi, and
// Gamma-scaled hi/lo); the state pass (fp16 copy, rescale by the next chunk's
// decay); the epilogue O = d O1 + O2 and the gated RMSNorm (node gdn.norm),
// on other warps and, for part of the tokens, on the chain warps while MMA7
// runs, overlapping the next chunk's chain.  The chunk tiles arrive by TMA a
// chunk or more ahead.
//
// prefill_overlap_kernel: both parts in one cooperative launch, for few
// (sequence, value head) units; the sequential CTAs read a chunk's workspace
// outputs once the prep group that made them has set the item's flag.
//
// Rows of a chunk past its sequence's end carry beta = 0 and g = 0, so their
// columns of T B, T B D are zero: they add nothing to U, W, Delta or the state,
// whatever finite values the staged rows hold there.
#include <cuda.h>

#include "chunk_math.cuh"
#include "gdn_device.cuh"
#include "launch.h"
#include "tma_host.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;
using namespace chunk;
using bf16 = __nv_bfloat16;

constexpr int kRawRows = kC + 3;                   // a chunk's rows plus the three before it
constexpr uint32_t kRawBlock = kRawRows * kD * 2;  // 17152 bytes

// ---- work geometry -----------------------------------------------------------
// Chunk slots index the workspace: fixed length, slot = b * nch + n; packed
// sequences, slot = (cu[b] >> 6) + b + n, which never collides (a sequence
// starting at token s with L tokens uses slots (s >> 6) + b .. (s >> 6) + b +
// ceil(L/64) - 1, below the next sequence's first slot).
struct ChunkLoc {
  int b, n, bos, len;
  bool ok;
};

__device__ __forceinline__ ChunkLoc locate(const SplitArgs &s, int slot) {
  ChunkLoc c{0, 0, 0, 0, false};
  if (!s.cu) {
    c.b = slot / s.nch;
    c.n = slot - c.b * s.nch;
    c.bos = c.b * s.T;
    c.len = s.T;
    c.ok = c.b < s.B;
    return c;
  }
  int lo = 0, hi = s.B - 1;  // the last sequence whose first slot is <= slot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((s.cu[mid] >> 6) + mid <= slot) lo = mid; else hi = mid - 1;
  }
  const int s0 = s.cu[lo], s1 = s.cu[lo + 1];
  if (s0 < 0 || s1 < s0 || s1 > s.T) return c;  // unusable offsets: the sequential kernel reports them
  c.b = lo;
  c.bos = s0;
  c.len = s1 - s0;
  c.n = slot - ((s0 >> 6) + lo);
  c.ok = c.n >= 0 && kC * c.n < c.len;
  return c;
}
__device__ __forceinline__ int slot_of(const SplitArgs &s, int b, int bos, int n) {
  return s.cu ? (bos >> 6) + b + n : b * s.nch + n;
}

// Non-blocking probe of an mbarrier phase.
__device__ __forceinline__ bool bar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// A plain bulk copy global -> shared completing on `bar` (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// =============================================================================
// prefill_prep_kernel
// =============================================================================
constexpr int kPrepThreads = 256;
// Shared memory (offsets from a 1024-aligned base).
constexpr uint32_t P_KQ = 0;        // [K;Q] K-major 128 x 128 fp16 (k^ hi rows 0-63, q^ rows 64-127)  32 KB
constexpr uint32_t P_TU = 32768;    // T diag(beta) hi  K-major [i][j]                                      8 KB
constexpr uint32_t P_TUL = 40960;   // T diag(beta) lo                                                      8 KB
constexpr uint32_t P_TW = 49152;    // -T diag(beta d)                                                      8 KB
constexpr uint32_t P_M = 57344;     // M fp16 K-major [i][j]                                                8 KB
constexpr uint32_t P_NW = P_TU;     // after MMA U / W: -W^T fp16 MN-major [k][j] over TU + TUL            16 KB
constexpr uint32_t P_UB0 = P_TW;    // after MMA U / W: U^T box 0 over TW + M                              16 KB
constexpr uint32_t P_RAW = 65536;   // raw v rows bf16 [67][128]; then L fp32 [64][68]                     17 KB
constexpr uint32_t P_TF = P_RAW + 64 * kLs * 4;  // T fp32 [64][64] (tfi); then U^T box 1                16 KB
constexpr uint32_t P_PB = P_TF + 16384;          // solve block products                                 4 KB
constexpr uint32_t P_VEC = P_PB + 4096;
struct PrepShared {
  ChunkVecs cv[2];  // the group's k-th item uses cv[k & 1]; the next item's are formed meanwhile
  uint64_t bar_kq, bar_raw, bar_qk, bar_uw;
  uint32_t tmem;
  int abort;
};
constexpr uint32_t kPrepSmem = P_VEC + ((sizeof(PrepShared) + 127) / 128) * 128 + 1024;
static_assert(64 * kLs * 4 >= kRawBlock, "the raw v region holds L");
static_assert(P_UB0 % 1024 == 0 && P_M == P_UB0 + 8192 && P_TF % 1024 == 0 && P_PB % 16 == 0 && P_VEC % 16 == 0,
              "alignment (U^T boxes: 1024)");
static_assert(kPrepSmem <= 113 * 1024, "two CTAs per SM");
// TMEM columns (256 allocated).
constexpr uint32_t TP_KQ = 0;    // [K K^T; Q K^T]                    64
constexpr uint32_t TP_V = 64;    // V^T fp16 pairs: hi 64..95, lo 96..127
constexpr uint32_t TP_U = 128;   // U^T [v][i]                        64
constexpr uint32_t TP_W = 192;   // -W^T [k][i]                       64
constexpr uint32_t kPrepTmem = 256;
constexpr int kBarSolve = 1;  // a prep group's solve barrier (the second group: 3)
constexpr int kBarPrep = 2;   // a prep group's own barrier (the second group: 4)
constexpr int kLoadTid = 160;   // warp 5, lane 0: a group's TMA loads
constexpr int kStoreTid = 192;  // warp 6, lane 0: a group's workspace stores and flags
constexpr int kGateWarp = 7;    // a group's gates and chunk vectors

// A prep group: 256 threads (8 warps) with their own kPrepSmem of shared
// memory, 256 TMEM columns and named barriers, taking work items first,
// first + step, ...  Without flags (prefill_prep_kernel) the items are the
// workspace's own order (slot * Hv + h, packed slots skipped where no chunk
// lies); with flags (prefill_overlap_kernel, fixed length only) they are
// walked chunk by chunk, (n, b, h), so that the sequential CTAs of the same
// launch find their next chunk early, and each item's flag is set once its
// outputs have landed in the workspace.
struct PrepGroup {
  uint8_t *sm;       // 1024-aligned
  uint32_t tmem;     // first of the group's 256 columns
  int tid;           // 0..255
  int bar, bar_solve;
  long long first, step;
  int *flags;
};
__device__ __forceinline__ void group_sync(const PrepGroup &G) { named_sync(G.bar, kPrepThreads); }
__device__ __forceinline__ bool group_sync_or(const PrepGroup &G, bool p) {
  return named_sync_or(G.bar, kPrepThreads, p);
}
// Release of an item's flag: its stores (TMA and plain) are complete and
// visible at GPU scope before the flag is.  The plain stores of the group's
// other threads precede it through the group barriers they passed, which the
// release (cumulative) covers.
__device__ __forceinline__ void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// The next item's tiles and gates are requested while the current one is
// computed: its q^ rows during the solve (MMA1 is done with them), its raw v
// rows once the solve is done with L (their space), its k^ rows once MMA W is
// done; its chunk vectors are formed while MMA U / W runs.  The loads belong
// to one thread of warp 5, the workspace stores (and, with flags, their
// completion and the flag) to one of warp 6: issuing a copy holds its warp a
// while, and neither warp has a part in the first step of the solve, nor
// warp 5 in writing the chunk vectors, where they issue.
template <bool kRawGates>
__device__ __forceinline__ void prep_role(const PrefillArgs &a, const SplitArgs &s, const CUtensorMap *tm_qkv,
                                          const CUtensorMap *tm_qk, const CUtensorMap *tm_u, const CUtensorMap *tm_nw,
                                          const CUtensorMap *tm_m, const PrepGroup &G) {
  uint8_t *sm = G.sm;
  PrepShared &V = *reinterpret_cast<PrepShared *>(sm + P_VEC);
  const Dims d = a.d;
  const int tid = G.tid, lane = threadIdx.x & 31, warp = tid >> 5;
  const int quad = warp & 3, half = warp >> 2;
  const int lrow = 32 * quad + lane;  // TMEM lane of this thread
  const uint32_t sbase = smem_u32(sm);
  const SolveSmem ss{reinterpret_cast<const float *>(sm + P_RAW), reinterpret_cast<float *>(sm + P_TF),
                     reinterpret_cast<float *>(sm + P_PB), sm + P_TU, sm + P_TUL, sm + P_TW};
  const bf16 *conv_w = static_cast<const bf16 *>(a.conv_w);
  const bf16 *conv0 = static_cast<const bf16 *>(a.conv0);
  const int r = d.Hv / d.Hk;
  const long long C = d.C;
  const long long nitems = (long long)s.nslots * d.Hv;
  const long long cv0 = 2LL * d.Hk * kD;  // first v channel

  if (tid == 0) {
    bar_init(&V.bar_kq, 1);
    bar_init(&V.bar_raw, 1);
    bar_init(&V.bar_qk, 1);
    bar_init(&V.bar_uw, 1);
    V.abort = 0;
  }
  zero_T_upper(ss, tid, kPrepThreads, 0, 3 * 192);
  fence_before();
  group_sync(G);
  fence_after();
  const uint32_t tmem = G.tmem;
  const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
  const uint32_t id_kk = idesc(128, 64, 0, 0), id_mk = idesc(128, 64, 1, 0);
  uint32_t ph_kq = 0, ph_raw = 0, ph_qk = 0, ph_uw = 0;
  bool q_req = false, k_req = false, raw_pending = false;  // kLoadTid: loads in flight
  bool stores = false;  // kStoreTid: stores issued
  long long pub = -1;   // kStoreTid: the item whose outputs are in flight, flagged once they land
  bool first = true;

  // Step `it` of the walk: its workspace item and chunk.  Steps and items
  // are below 2^24 (the host's limit), so the divisions are 32-bit.
  const unsigned hv = (unsigned)d.Hv;
  auto head_of = [&](long long it) -> int { return (int)((unsigned)it % hv); };
  auto resolve = [&](long long it, ChunkLoc &c) -> long long {
    if (!G.flags) {
      c = locate(s, (int)((unsigned)it / hv));
      return it;
    }
    const unsigned bh = (unsigned)s.B * hv;
    const unsigned n = (unsigned)it / bh, rem = (unsigned)it - n * bh, b = rem / hv, h = rem - b * hv;
    c = ChunkLoc{(int)b, (int)n, (int)b * s.T, s.T, true};
    return ((long long)b * s.nch + n) * d.Hv + h;
  };
  // The next step at or after `it` with a valid chunk (every thread computes the same).
  auto next_valid = [&](long long it, ChunkLoc &c, long long &itm) -> long long {
    for (; it < nitems; it += G.step) {
      itm = resolve(it, c);
      if (c.ok) return it;
    }
    return nitems;
  };
  // kStoreTid: the flag of the item in flight once its outputs have landed
  // (keep_newest: the most recent store group may still be in flight).
  auto publish = [&](bool keep_newest) {
    if (pub >= 0) {
      if (keep_newest) bulk_wait_all_but_one();
      else bulk_wait_all();
      fence_proxy_async_all();
      __threadfence();
      st_release_gpu(G.flags + pub, 1);
      pub = -1;
    }
  };
  // kLoadTid: an item's q^ rows (rows 64-127 of [K;Q]) and k^ hi rows (rows
  // 0-63) complete one phase of bar_kq: the first part only announces its
  // bytes, the second arrives.  The raw v rows complete bar_raw.
  auto load_kq_part = [&](long long it, const ChunkLoc &c, int plane) {
    const int kh = head_of(it) / r;
#pragma unroll
    for (int at = 0; at < 2; ++at)
      tma_load_3d(sbase + P_KQ + at * 16384 + (plane == 0 ? 64 * 128 : 0), tm_qk, kh * kD + 64 * at, c.bos + kC * c.n,
                  plane, &V.bar_kq);
  };
  auto request_q = [&](long long it, const ChunkLoc &c) {
    bar_expect_tx_only(&V.bar_kq, kC * kD * 2);
    load_kq_part(it, c, 0);
    q_req = true;
  };
  auto request_k = [&](long long it, const ChunkLoc &c) {
    bar_expect_tx(&V.bar_kq, kC * kD * 2);
    load_kq_part(it, c, 1);
    k_req = true;
  };
  auto request_raw = [&](long long it, const ChunkLoc &c) {
    bar_expect_tx(&V.bar_raw, kRawBlock);
    tma_load_3d(sbase + P_RAW, tm_qkv, (int)(cv0 + head_of(it) * kD), c.bos + kC * c.n - 3, 0, &V.bar_raw);
    raw_pending = true;
  };
  // kGateWarp: an item's gates (raw bf16 bits for raw projections), requested
  // an item before its chunk vectors are formed.
  float gv[2] = {0.f, 0.f}, bv[2] = {0.f, 0.f}, nea = 0.f, dtb = 0.f;
  auto load_gates = [&](long long it, const ChunkLoc &c) {
    const int h = head_of(it);
    load_gb<kRawGates>(a.gate, c.bos, d.Hv, h, kC * c.n, c.len, lane, gv, bv);
    if (kRawGates) {
      nea = a.gate.A_log[h];
      dtb = a.gate.dt_bias[h];
    }
  };
  auto form_vectors = [&](const ChunkLoc &c, ChunkVecs &cvd) {
    finish_gb<kRawGates>(kRawGates ? -expf(nea) : 0.f, dtb, kC * c.n, c.len, lane, gv, bv);
    chunk_vectors(cvd, gv, bv, lane);
  };

  ChunkLoc c{};
  long long item = 0;
  long long it = next_valid(G.first, c, item);
  if (it < nitems) {
    if (tid == kLoadTid) {
      request_q(item, c);
      request_k(item, c);
      request_raw(item, c);
    }
    if (warp == kGateWarp) {  // the first item's chunk vectors; the second item's gates
      load_gates(item, c);
      form_vectors(c, V.cv[0]);
      ChunkLoc c2{};
      long long item2 = 0;
      if (next_valid(it + G.step, c2, item2) < nitems) load_gates(item2, c2);
    }
  }
  for (int k = 0; it < nitems; ++k) {
    const ChunkVecs &CV = V.cv[k & 1];
    const int h = head_of(item);
    const int t0 = kC * c.n, T = c.len;
    const long long cv = cv0 + (long long)h * kD;
    ChunkLoc cn{};
    long long next = 0;
    const long long it_next = next_valid(it + G.step, cn, next);
    const bool more = it_next < nitems;
    __syncwarp();
    const bool kq_ok = bar_wait(&V.bar_kq, ph_kq);
    const bool raw_ok = kq_ok && bar_wait(&V.bar_raw, ph_raw);
    if (kq_ok) {
      ph_kq ^= 1u;
      if (tid == kLoadTid) q_req = k_req = false;
    }
    if (raw_ok) {
      ph_raw ^= 1u;
      if (tid == kLoadTid) raw_pending = false;
    }
    bool ok = raw_ok;
    if (group_sync_or(G, !ok)) {
      if (tid == 0) {
        atomicOr(a.err, kErrTimeout);
        V.abort = 1;
      }
      break;
    }
    if (c.n == 0) {  // rows before the sequence's first token: the carried window, or zeros
      if (tid < 48) {
        const int rw = tid >> 4, g8 = tid & 15;
        *reinterpret_cast<uint4 *>(sm + P_RAW + 256 * rw + 16 * g8) =
            conv0 ? *reinterpret_cast<const uint4 *>(conv0 + ((long long)c.b * 3 + rw) * C + cv + 8 * g8)
                  : make_uint4(0u, 0u, 0u, 0u);
      }
      group_sync(G);
    }
    // MMA1 (warp 0): [K;Q] K^T -> K K^T (lanes 0-63), Q K^T (lanes 64-127)
    const uint32_t kq = sbase + P_KQ;
    if (warp == 0) {
      fence_after();
      issue_w(tmem + TP_KQ, id_kk, 8, false, [&](int ks) { return desc_k(kq, ks, 128); },
              [&](int ks) { return desc_k(kq, ks, 128); });
      commit_w(&V.bar_qk);
    }
    // The v tiles (every warp): row v = lrow, tokens 32 half .. 32 half + 31;
    // conv + SiLU, zero past the sequence, fp16 hi/lo pairs into TMEM (the A
    // operand of MMA U: lane = v, column c = tokens 2c, 2c + 1).  Pairs of
    // tokens on the paired fp32 pipes.
    {
      const bf16 *raw = reinterpret_cast<const bf16 *>(sm + P_RAW) + lrow;
      const float4 w4 = ld_io4(conv_w + 4 * (cv + lrow));
      const float2 w0 = make_float2(w4.x, w4.x), w1 = make_float2(w4.y, w4.y), w2 = make_float2(w4.z, w4.z),
                   w3 = make_float2(w4.w, w4.w);
      const int j0 = 32 * half;
      const bool tail = t0 + kC > T;  // the sequence ends inside this chunk
      float2 xa = make_float2(__bfloat162float(raw[(j0 + 0) * kD]), __bfloat162float(raw[(j0 + 1) * kD]));
      float2 xb = make_float2(__bfloat162float(raw[(j0 + 2) * kD]), __bfloat162float(raw[(j0 + 3) * kD]));
      uint32_t wh[16], wl[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int j = j0 + 2 * q;  // tokens j, j + 1 use rows j .. j + 4
        const float2 xc = make_float2(__bfloat162float(raw[(j + 4) * kD]), __bfloat162float(raw[(j + 5 < kRawRows ? j + 5 : j + 4) * kD]));
        float2 acc = __fmul2_rn(w0, xa);
        acc = __ffma2_rn(w1, make_float2(xa.y, xb.x), acc);
        acc = __ffma2_rn(w2, xb, acc);
        acc = __ffma2_rn(w3, make_float2(xb.y, xc.x), acc);
        float2 u = silu2(acc);
        if (tail) {
          if (t0 + j >= T) u.x = 0.f;
          if (t0 + j + 1 >= T) u.y = 0.f;
        }
        split2(u.x, u.y, wh[q], wl[q]);
        xa = xb;
        xb = xc;
      }
      tmem_st16w_nw(tl + TP_V + 16 * half, wh);
      tmem_st16w_nw(tl + TP_V + 32 + 16 * half, wl);
      tmem_wait_st();
    }
    // The previous item's stores must have read their sources (M, the T tiles
    // and the T scratch are written next).
    if (tid == kStoreTid && stores) bulk_wait_read();
    fence_before();
    group_sync(G);  // the v rows are read: L may take their space
    ok = bar_wait(&V.bar_qk, ph_qk);
    ph_qk ^= 1u;
    fence_after();
    if (group_sync_or(G, !ok)) {
      if (tid == 0) {
        atomicOr(a.err, kErrTimeout);
        V.abort = 1;
      }
      break;
    }
    // L (fp32, strictly lower, decayed beta K K^T) and M (fp16, decayed Q K^T incl. the diagonal)
    {
      float v[32], rr[32];
      tmem_ld32(tl + TP_KQ + 32 * half, v);
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
        float *L = reinterpret_cast<float *>(sm + P_RAW) + i * kLs + j0;
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float2 p01 =
              __fmul2_rn(__fmul2_rn(make_float2(bi, bi), make_float2(v[q], v[q + 1])), make_float2(rr[q], rr[q + 1]));
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
        for (int q = 0; q < 4; ++q) st_h8_inrange(sm + P_M + kmaj(i, j0 + 8 * q, kC), v + 8 * q);  // |M| <= q_scale
      }
    }
    fence_smem_to_async();
    group_sync(G);  // L and M written
    if (tid == kStoreTid) {
      tma_store_2d(tm_m, sbase + P_M, 0, (int)(item * kC));
      bulk_commit();
      stores = true;
    }
    // T = (I + L)^{-1} and the fp16 tiles (their upper blocks are zeroed
    // again: the previous item's -W^T and U^T staging used their space).
    // Meanwhile (the diagonal blocks) the store thread sets the previous
    // item's flag once its outputs have landed (with flags), and the next
    // item's q^ rows are requested (MMA1 is long done with them).
    solve_T(ss, CV, tid, G.bar_solve, true, [&]() {
      if (tid == kStoreTid && G.flags) publish(true);
      if (tid == kLoadTid && more) request_q(next, cn);
    });
    fence_smem_to_async();
    fence_before();
    group_sync(G);
    // MMA U (hi*hi + lo*hi + hi*lo, A = V^T from TMEM) and MMA W (warp 0).
    if (warp == 0) {
      fence_after();
      auto b_tu = [&](int ks) { return desc_k(sbase + P_TU, ks, kC); };
      issue_ta_w(tmem + TP_U, tmem + TP_V, id_kk, 4, false, b_tu);
      issue_ta_w(tmem + TP_U, tmem + TP_V + 32, id_kk, 4, true, b_tu);
      issue_ta_w(tmem + TP_U, tmem + TP_V, id_kk, 4, true, [&](int ks) { return desc_k(sbase + P_TUL, ks, kC); });
      issue_w(tmem + TP_W, id_mk, 4, false, [&](int ks) { return desc(kq + (uint32_t)(ks * 2048), 128 * 128, 1024); },
              [&](int ks) { return desc_k(sbase + P_TW, ks, kC); });
      commit_w(&V.bar_uw);
    }
    if (tid < 2 * kC) {  // the chunk vectors d and Gamma, fp32 [2][64]
      float *vec = s.ws_vec + item * (2 * kC);
      // (ordered before the item's flag by the group barriers that precede
      // the store thread's release; no fence of its own)
      if (in_bounds(item * (2 * kC) + tid + 1, nitems * (2 * kC), a.err)) vec[tid] = tid < kC ? CV.d[tid] : CV.gam[tid - kC];
    }
    if (tid == kLoadTid && more) request_raw(next, cn);  // L is done with: the next item's raw v rows may land
    if (warp == kGateWarp && more) {  // the next item's chunk vectors; the gates of the one after it
      form_vectors(cn, V.cv[(k + 1) & 1]);
      ChunkLoc c2{};
      long long item2 = 0;
      if (next_valid(it_next + G.step, c2, item2) < nitems) load_gates(item2, c2);
    }
    __syncwarp();
    ok = bar_wait(&V.bar_uw, ph_uw);
    ph_uw ^= 1u;
    fence_after();
    if (group_sync_or(G, !ok)) {
      if (tid == 0) {
        atomicOr(a.err, kErrTimeout);
        V.abort = 1;
      }
      break;
    }
    // MMA W is done with the k^ rows: the next item's may land.  The M store
    // has long read its source (whose space takes U^T box 0).
    if (tid == kLoadTid && more) request_k(next, cn);
    if (tid == kStoreTid) bulk_wait_read();
    group_sync(G);
    {
      // U^T [v][i] fp32 -> staging box `half` (rows v, 32 values of 4 bytes, 128-byte swizzle)
      float v[32];
      tmem_ld32(tl + TP_U + 32 * half, v);
      uint8_t *box = sm + (half == 0 ? P_UB0 : P_TF) + lrow * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4 *>(box + ((q ^ (lrow & 7)) << 4)) =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      // -W^T [k][i] -> fp16 MN-major (the B operand layout of MMA4)
      tmem_ld32(tl + TP_W + 32 * half, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) st_h8_inrange(sm + P_NW + mnmaj(32 * half + 8 * q, lrow, kD), v + 8 * q);
    }
    fence_smem_to_async();
    fence_before();
    group_sync(G);
    if (tid == kStoreTid) {
      tma_store_2d(tm_u, sbase + P_UB0, 0, (int)(item * kD));
      tma_store_2d(tm_u, sbase + P_TF, 32, (int)(item * kD));
      tma_store_2d(tm_nw, sbase + P_NW, 0, (int)(item * kD));
      bulk_commit();
      if (G.flags) {
        pub = item;
        if (first) publish(false);  // the first items are the launch's first chunks: flag them without delay
      }
    }
    first = false;
    it = it_next;
    item = next;
    c = cn;
  }
  // Before the group ends: the stores complete (the last item flagged), no
  // load still lands (a q^ request alone completes its phase with an
  // arrival), and no MMA still writes TMEM (after an early exit).
  if (tid == kStoreTid) {
    bulk_wait_all();
    if (G.flags) publish(false);
  }
  if (tid == kLoadTid) {
    if (q_req && !k_req) mbar_arrive(&V.bar_kq);
    if (q_req || k_req) bar_wait(&V.bar_kq, ph_kq);
    if (raw_pending) bar_wait(&V.bar_raw, ph_raw);
  }
  fence_before();
  group_sync(G);
}

template <bool kRawGates>
__global__ void __launch_bounds__(kPrepThreads, 2)
    prefill_prep_kernel(const PrefillArgs a, const SplitArgs s, const __grid_constant__ CUtensorMap tm_qkv,
                        const __grid_constant__ CUtensorMap tm_qk, const __grid_constant__ CUtensorMap tm_u,
                        const __grid_constant__ CUtensorMap tm_nw, const __grid_constant__ CUtensorMap tm_m) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  PrepShared &V = *reinterpret_cast<PrepShared *>(sm + P_VEC);
  if (threadIdx.x < 32) tmem_alloc(&V.tmem, kPrepTmem);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = V.tmem;
  const PrepGroup G{sm, tmem, (int)threadIdx.x, kBarPrep, kBarSolve, (long long)blockIdx.x, (long long)gridDim.x,
                    nullptr};
  prep_role<kRawGates>(a, s, &tm_qkv, &tm_qk, &tm_u, &tm_nw, &tm_m, G);
  fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    fence_after();
    tmem_dealloc(tmem, kPrepTmem);
  }
}

// =============================================================================
// prefill_seq_kernel
// =============================================================================
// Warps 0-6: the epilogue (O staging, the gated norm of most tokens); warp 7:
// the TMA producer (the U^T tiles and chunk stages, the flags and decays), in
// one converged loop; warps 8-15: the chain (the state-dependent MMAs, issued
// by warp 8, and the Delta and state passes, two warps per TMEM lane quadrant,
// each on half of the columns; warps 9-15 also form the gated norm of the
// other tokens while MMA7 runs, and reload the z rows).
constexpr int kSeqThreads = 512;
constexpr int kProducerWarp = 7;
constexpr int kEpiThreads = 224;
constexpr int kChainThreads = 256;
constexpr int kIssuerTid = 256;  // warp 8, lane 0
// One stage (a chunk's tiles), offsets within the stage; fp16, 128-byte swizzle.
constexpr uint32_t Q_Q = 0;         // q^ K-major [i][k] (64 rows, k halves 8 KB apart)   16 KB
constexpr uint32_t Q_KH = 16384;    // k^ hi [j][k]                                       16 KB
constexpr uint32_t Q_KL = 32768;    // k^ lo [j][k]                                       16 KB
constexpr uint32_t Q_NW = 49152;    // -W^T MN-major [k][j]                               16 KB
constexpr uint32_t Q_M = 65536;     // M K-major [i][j]                                    8 KB
constexpr uint32_t kStage = 73728;
constexpr uint32_t kStageTx = 3 * 16384 + 16384 + 8192 + 2 * kC * 4;  // tiles + the vectors
constexpr uint32_t S_U = 2 * kStage;          // U^T fp32, two boxes [128 v][32] (128-byte swizzle)  32 KB
constexpr uint32_t S_Z = S_U + 32768;         // z rows bf16 [64][128]                                16 KB
constexpr uint32_t S_OST = S_Z + 16384;       // O staging fp32 [64 i][128 v]                         32 KB
constexpr uint32_t S_VEC = S_OST + 32768;     // d, Gamma of the two stages, fp32 [2][2][64]            1 KB
constexpr uint32_t S_BAR = S_VEC + 1024;
struct SeqShared {
  uint64_t full[2];    // a stage's tiles and vectors landed
  uint64_t bar_u;      // U^T landed
  uint64_t bar_z;      // z rows landed
  uint64_t bar_d;      // MMA4 done
  uint64_t bar_o;      // MMA5 and MMA6 done
  uint64_t bar_s;      // MMA7 done
  uint64_t bar_ufree;  // the chain has read U^T (one arrival per chunk)
  uint64_t bar_ofree;  // the epilogue has staged O1, O2 (one arrival per chunk): TMEM's O is free
  uint64_t bar_end;
  uint32_t tmem;
  int abort;
  int req_full[2], req_u, req_z;  // requests issued (each completes one phase)
  int ahead;                      // chunks 0 .. ahead-1: flags seen (when given) and decays in dcr
  int s_seen;                     // chunks whose MMA7 (and the MMAs issued before it) are done
  int epi_seen;                   // chunks whose MMA6 is done and whose vectors the epilogue has read
  int epi_zread;                  // chunks whose staged O and z rows 0..kEpiTokens-1 the epilogue has read
  int help_loaded;                // chunks whose staged O and z rows kEpiTokens.. the chain warps have read
  alignas(16) float de[2][64];    // the epilogue's copy of chunk n's d at n & 1 (read as float4)
  float dcr[16];                  // e^{G_last} of chunk m at m % 16
};
constexpr uint32_t kSeqSmem = S_BAR + ((sizeof(SeqShared) + 127) / 128) * 128 + 1024;
static_assert(offsetof(SeqShared, de) % 16 == 0 && S_BAR % 16 == 0, "16-byte loads of the d copy");
static_assert(kSeqSmem <= 232448, "shared memory per CTA");
static_assert(S_U % 1024 == 0 && S_Z % 128 == 0 && kStage % 1024 == 0, "TMA destinations");
// TMEM columns (512 allocated).
constexpr uint32_t TS_S = 0;      // state fp32 [v][k]                  128
constexpr uint32_t TS_O1 = 128;   // S Q^T [v][i]                        64
constexpr uint32_t TS_O2 = 192;   // Delta^T M^T [v][i]                  64
constexpr uint32_t TS_D = 256;    // S (-W^T) [v][j]                     64
constexpr uint32_t TS_DG = 320;   // (Delta Gamma)^T fp16: hi 320..351, lo 352..383
constexpr uint32_t TS_DH = 384;   // Delta^T fp16 hi                     32
constexpr uint32_t TS_S16 = 448;  // state fp16 pairs [v][k/2]           64
constexpr uint32_t kSeqTmem = 512;
constexpr int kBarChain = 2;  // warps 8-15
constexpr int kBarEpi = 3;    // warps 0-6
constexpr int kBarHelp = 4;   // warps 9-15 (the chain warps that do not issue MMAs)
constexpr int kHelpThreads = 224;
constexpr int kHelpLeadTid = 288;  // warp 9, lane 0
// The gated norm's tokens: 0 .. kEpiTokens-1 by the epilogue's 14 half-warps,
// the rest by the 14 half-warps of chain warps 9-15.
constexpr int kEpiTokens = 40;
constexpr int kEpiNR = (kEpiTokens + 13) / 14, kHelpNR = (kC - kEpiTokens + 13) / 14;

__device__ __forceinline__ bool seq_aborted(const SeqShared &V) { return *reinterpret_cast<const volatile int *>(&V.abort) != 0; }
// Bounded wait (about one second) for a shared counter to reach `m`, then
// ordered before what follows.
__device__ __forceinline__ bool count_wait(int *p, int m) {
  const volatile int *v = p;
  if (*v < m) {
    const uint64_t t0 = global_ns();
    while (*v < m) {
      if (global_ns() - t0 > 1000000000ull) return false;
      __nanosleep(32);
    }
  }
  __threadfence_block();
  return true;
}
// The stage producer has covered `m` chunks (V.ahead >= m).
__device__ __forceinline__ bool ahead_wait(SeqShared &V, int m) { return count_wait(&V.ahead, m); }
__device__ __forceinline__ void seq_fail(SeqShared &V, unsigned int *err) {
  atomicOr(err, kErrTimeout);
  *reinterpret_cast<volatile int *>(&V.abort) = 1;
}

// The gated RMSNorm (node gdn.norm) of NR tokens i0, i0 + di, ... of the chunk,
// one half-warp per token; lane hl of the half-warp takes channels 4 hl .. 4 hl
// + 3 and 64 + 4 hl .. 64 + 4 hl + 3 (16-byte reads of the staged rows without
// bank conflicts).  norm_load takes the staged O and z rows into registers
// (after it the z buffer may be refilled); norm_store forms y for every slot
// without branches (a slot past the chunk holds zeros and gives y = 0; the
// tokens stay independent for the scheduler) and writes o for valid tokens.
template <int NR>
struct NormRegs {
  float4 o0[NR], o1[NR];
  uint2 z0[NR], z1[NR];
};
template <int NR>
__device__ __forceinline__ void norm_load(const uint8_t *sm, NormRegs<NR> &R, int nv, int i0, int di, int lane) {
  const float *ost = reinterpret_cast<const float *>(sm + S_OST);
  const int hl = lane & 15;
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int i = i0 + di * m;
    R.o0[m] = R.o1[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    R.z0[m] = R.z1[m] = make_uint2(0u, 0u);
    if (i < nv) {
      R.o0[m] = ld4(ost + i * kD + 4 * hl);
      R.o1[m] = ld4(ost + i * kD + 64 + 4 * hl);
      R.z0[m] = *reinterpret_cast<const uint2 *>(sm + S_Z + i * kD * 2 + 8 * hl);
      R.z1[m] = *reinterpret_cast<const uint2 *>(sm + S_Z + i * kD * 2 + 128 + 8 * hl);
    }
  }
}
__device__ __forceinline__ void widen2(uint2 u, float2 (&v)[2]) {
  v[0] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
  v[1] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
}
template <int NR>
__device__ __forceinline__ void norm_store(const NormRegs<NR> &R, const bf16 *norm_w, bf16 *o, const Dims &d,
                                           long long bos, int h, int t0, int nv, int i0, int di, int lane,
                                           long long o_size, unsigned int *err) {
  const int hl = lane & 15;
  float2 wn[4];
  widen2(*reinterpret_cast<const uint2 *>(norm_w + 4 * hl), *reinterpret_cast<float2(*)[2]>(&wn[0]));
  widen2(*reinterpret_cast<const uint2 *>(norm_w + 64 + 4 * hl), *reinterpret_cast<float2(*)[2]>(&wn[2]));
  bf16 *ob = o + ((bos + t0) * d.Hv + h) * kD + 4 * hl;
  const long long ostride = (long long)d.Hv * kD;
#pragma unroll
  for (int m = 0; m < NR; ++m) {
    const int i = i0 + di * m;
    float ss = dot4(R.o0[m], R.o0[m]) + dot4(R.o1[m], R.o1[m]);
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rstd = rsqrtf(ss * (1.0f / kD) + d.eps_norm);
    float2 zz[4];
    widen2(R.z0[m], *reinterpret_cast<float2(*)[2]>(&zz[0]));
    widen2(R.z1[m], *reinterpret_cast<float2(*)[2]>(&zz[2]));
    const float2 op[4] = {make_float2(R.o0[m].x, R.o0[m].y), make_float2(R.o0[m].z, R.o0[m].w),
                          make_float2(R.o1[m].x, R.o1[m].y), make_float2(R.o1[m].z, R.o1[m].w)};
    uint32_t yw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 sg = silu2(zz[q]);
      const float2 y = __fmul2_rn(__fmul2_rn(wn[q], __fmul2_rn(op[q], make_float2(rstd, rstd))), sg);
      __nv_bfloat162 t = __floats2bfloat162_rn(y.x, y.y);
      yw[q] = *reinterpret_cast<uint32_t *>(&t);
    }
    bf16 *orow = ob + i * ostride;
    if (i < nv && in_bounds((orow - o) + 68, o_size, err)) {
      *reinterpret_cast<uint2 *>(orow) = make_uint2(yw[0], yw[1]);
      *reinterpret_cast<uint2 *>(orow + 64) = make_uint2(yw[2], yw[3]);
    }
  }
}

// The sequential part for the CTA's (sequence, value head), run by the whole
// CTA (kSeqThreads threads).  With flags (prefill_overlap_kernel) a chunk's
// workspace outputs are used only once its flag is set.
__device__ __forceinline__ void seq_role(const PrefillArgs &a, const SplitArgs &s, const CUtensorMap *tm_qk,
                                         const CUtensorMap *tm_z, const CUtensorMap *tm_u, const CUtensorMap *tm_nw,
                                         const CUtensorMap *tm_m, uint8_t *sm, const int *flags) {
  SeqShared &V = *reinterpret_cast<SeqShared *>(sm + S_BAR);
  const Dims d = a.d;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x % d.Hv;
  int b = blockIdx.x / d.Hv;
  const int r = d.Hv / d.Hk, kh = h / r;
  const long long C = d.C;
  const uint32_t sbase = smem_u32(sm);
  if (a.cu_seqlens && d.B <= kLongestFirstMax)  // packed: the longest sequences first
    b = longest_first(a.cu_seqlens, d.B, b, reinterpret_cast<int *>(sm + S_OST));
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
  const long long unit_off = ((long long)b * d.Hv + h) * kD * kD;
  const long long S_size = (long long)d.B * d.Hv * kD * kD;                                        // S_T elements
  const long long o_size = (a.cu_seqlens ? (long long)d.T : (long long)d.B * d.T) * d.Hv * kD;  // o elements
  const bf16 *x = static_cast<const bf16 *>(a.qkv_pre) + bos * C;
  const bf16 *conv0 = a.conv0 ? static_cast<const bf16 *>(a.conv0) + (long long)b * 3 * C : nullptr;
  const int cq = kh * kD, ck = d.Hk * kD + kh * kD, cvv = 2 * d.Hk * kD + h * kD;

  // The carried conv window: the last three raw rows of the channels this CTA owns.
  auto write_conv_T = [&]() {
    bf16 *cT = static_cast<bf16 *>(a.conv_T) + (long long)b * 3 * C;
    const bool own_qk = (h % r) == 0;
    for (int idx = tid; idx < 3 * 3 * kD; idx += kSeqThreads) {
      const int e = idx / (3 * kD), rem = idx % (3 * kD), blk = rem / kD, ch = rem % kD;
      if (blk < 2 && !own_qk) continue;
      const long long cc = (blk == 0 ? cq : blk == 1 ? ck : cvv) + ch;
      const int t = T - 3 + e;
      bf16 val;
      if (t >= 0) val = x[(long long)t * C + cc];
      else if (conv0) val = conv0[(long long)(3 + t) * C + cc];
      else val = bf16(0.f);
      if (in_bounds(((long long)b * 3 + e) * C + cc + 1, (long long)d.B * 3 * C, a.err)) cT[(long long)e * C + cc] = val;
    }
  };
  if (T == 0) {  // an empty packed sequence: state and window pass through
    float4 *dst = reinterpret_cast<float4 *>(a.S_T + unit_off);
    const float4 *src = a.S0 ? reinterpret_cast<const float4 *>(a.S0 + unit_off) : nullptr;
    if (src != dst)
      for (int i = tid; i < kD * kD / 4; i += kSeqThreads)
        if (in_bounds(unit_off + 4 * i + 4, S_size, a.err)) dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    write_conv_T();
    return;
  }
  const int nch = (T + kC - 1) / kC;
  auto item_of = [&](int n) -> long long { return (long long)slot_of(s, b, (int)bos, n) * d.Hv + h; };

  if (tid == 0) {
    bar_init(&V.full[0], 1);
    bar_init(&V.full[1], 1);
    bar_init(&V.bar_u, 1);
    bar_init(&V.bar_z, 1);
    bar_init(&V.bar_d, 1);
    bar_init(&V.bar_o, 1);
    bar_init(&V.bar_s, 1);
    bar_init(&V.bar_ufree, 1);
    bar_init(&V.bar_ofree, 1);
    bar_init(&V.bar_end, 1);
    V.abort = 0;
    V.req_full[0] = V.req_full[1] = V.req_u = V.req_z = 0;
    V.ahead = V.s_seen = V.epi_seen = V.epi_zread = V.help_loaded = 0;
  }
  if (warp == 0) tmem_alloc(&V.tmem, kSeqTmem);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = V.tmem;
  auto vec_d = [&](int st) { return reinterpret_cast<const float *>(sm + S_VEC + 512 * st); };  // d [64], Gamma [64]

  // The z rows are reloaded by the chain warps once both parts of the gated
  // norm have read them (chunk 0's by the epilogue); the stages, the U^T
  // tiles, the flags and the decays by the producer warp, in one ordered loop
  // (no warp runs diverged waits).
  auto load_z = [&](int n) {  // one thread
    bar_expect_tx(&V.bar_z, kC * kD * 2);
    tma_load_3d(sbase + S_Z, tm_z, h * kD, (int)(bos + kC * n), 0, &V.bar_z);
    V.req_z = n + 1;
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------ the producer (warp 7)
    // Step n: U^T of chunk n once the chain has read chunk n-1's; then
    // V.ahead past chunk n+2 (its flag seen, with flags, and its decay in the
    // ring); then the stage of chunk n+1 into chunk n-1's buffer once
    // MMA7(n-1) and MMA6(n-1) are done and the epilogue has copied chunk
    // n-1's vectors.  The stage's two conditions are counters, not barrier
    // phases: while this warp waits for a flag the chain may finish another
    // chunk, and a phase two ahead would read as not yet complete.  A chunk's
    // workspace outputs are loaded only after its flag was seen.  Lane 0
    // issues; every wait is bounded.
    // V.ahead up to `need`: lanes 0-7 look at the next 8 chunks' flags at
    // once (with flags), and the leading run that is set is announced with
    // its decays, one round trip for up to 8 chunks.  The ring holds 16
    // decays and at most 10 are ahead of the chain's reads.
    auto advance = [&](int need) -> bool {
      int have = *reinterpret_cast<volatile int *>(&V.ahead);
      uint64_t t0 = 0;
      while (have < need) {
        const int m = have + lane;
        const bool mine = lane < 8 && m < nch;
        bool set = true;
        if (mine && flags) {
          int v;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flags + item_of(m)) : "memory");
          set = v != 0;
        }
        const unsigned run = __ballot_sync(0xffffffffu, !mine || set);
        const int cnt = min(min(__ffs(~run | 0x100u) - 1, 8), nch - have);
        if (cnt == 0) {
          if (t0 == 0) t0 = global_ns();
          else if (global_ns() - t0 > 1000000000ull) return false;
          __nanosleep(256);
          continue;
        }
        if (lane < cnt) V.dcr[m & 15] = s.ws_vec[item_of(m) * (2 * kC) + kC - 1];
        __syncwarp();
        have += cnt;
        if (lane == 0) {
          __threadfence_block();
          *reinterpret_cast<volatile int *>(&V.ahead) = have;
        }
        __syncwarp();
      }
      return true;
    };
    auto load_stage = [&](int m) {
      if (flags) fence_proxy_async_all();  // the outputs, released by a prep group, read by TMA
      if (lane == 0) {
        const int st = m & 1;
        const uint32_t sb = sbase + st * kStage;
        const long long it = item_of(m);
        uint64_t *bar = &V.full[st];
        bar_expect_tx(bar, kStageTx);
#pragma unroll
        for (int at = 0; at < 2; ++at) {
          tma_load_3d(sb + Q_Q + at * 8192, tm_qk, kh * kD + 64 * at, (int)(bos + kC * m), 0, bar);
          tma_load_3d(sb + Q_KH + at * 8192, tm_qk, kh * kD + 64 * at, (int)(bos + kC * m), 1, bar);
          tma_load_3d(sb + Q_KL + at * 8192, tm_qk, kh * kD + 64 * at, (int)(bos + kC * m), 2, bar);
        }
        tma_load_2d(sb + Q_NW, tm_nw, 0, (int)(it * kD), bar);
        tma_load_2d(sb + Q_M, tm_m, 0, (int)(it * kC), bar);
        bulk_load(sbase + S_VEC + st * 512, s.ws_vec + it * (2 * kC), 2 * kC * 4, bar);
        V.req_full[st] += 1;
      }
      __syncwarp();
    };
    auto load_u = [&](int m) {
      if (flags) fence_proxy_async_all();
      if (lane == 0) {
        const long long it = item_of(m);
        bar_expect_tx(&V.bar_u, 32768);
        tma_load_2d(sbase + S_U, tm_u, 0, (int)(it * kD), &V.bar_u);
        tma_load_2d(sbase + S_U + 16384, tm_u, 32, (int)(it * kD), &V.bar_u);
        V.req_u = m + 1;
      }
      __syncwarp();
    };
    bool good = advance(min(3, nch));
    if (good) {
      load_stage(0);
      load_u(0);
      if (nch > 1) load_stage(1);
    }
    for (int n = 1; good && n < nch; ++n) {
      good = __all_sync(0xffffffffu, bar_wait(&V.bar_ufree, (uint32_t)(n - 1) & 1u));
      if (!good || seq_aborted(V)) break;
      load_u(n);
      if (!(good = advance(min(n + 3, nch)))) break;  // meanwhile MMA7(n-1) and the epilogue go on
      if (n + 1 < nch) {  // chunk n+1 goes where chunk n-1 was, once that is done with
        good = __all_sync(0xffffffffu, count_wait(&V.s_seen, n) && count_wait(&V.epi_seen, n));
        if (!good || seq_aborted(V)) break;
        load_stage(n + 1);
      }
    }
    if (!good && lane == 0) seq_fail(V, a.err);
  } else if (warp >= 8) {
    // ------------------------------------------------ the chain (warps 8-15)
    const int quad = warp & 3, ch = (warp - 8) >> 2;  // lane quadrant; column half
    const int lrow = 32 * quad + lane;                // state row v of this thread
    const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
    const bool issuer = warp == 8;
    const uint32_t id_kk = idesc(128, 64, 0, 0), id_km = idesc(128, 64, 0, 1), id_km128 = idesc(128, 128, 0, 1);
    bool ok = true;
    // e^{G_last} of chunk m (the decay the state takes at its start): in the
    // ring once V.ahead > m, in practice a chunk or more before it is needed.
    auto dc_of = [&](int m) -> float {
      if (!ahead_wait(V, m + 1)) ok = false;
      return *reinterpret_cast<volatile const float *>(&V.dcr[m & 15]);
    };
    const float dc0 = dc_of(0);
    // Initial state: TMEM fp32 <- d_C(chunk 0) S0, fp16 copy <- S0 (this
    // thread: row lrow, columns 64 ch .. 64 ch + 63).
#pragma unroll 1
    for (int k0 = 64 * ch; k0 < 64 * ch + 64; k0 += 32) {
      float v[32];
      if (a.S0) {
        const float4 *src = reinterpret_cast<const float4 *>(a.S0 + unit_off + (long long)lrow * kD + k0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 f = src[q];
          v[4 * q] = f.x;
          v[4 * q + 1] = f.y;
          v[4 * q + 2] = f.z;
          v[4 * q + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = 0.f;
      }
      uint32_t w16[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) w16[q] = pack2_sat(v[2 * q], v[2 * q + 1]);
      tmem_st16w_nw(tl + TS_S16 + k0 / 2, w16);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] *= dc0;
      tmem_st32(tl + TS_S + k0, v);
    }
    tmem_wait_st();
    fence_before();
    named_sync(kBarChain, kChainThreads);
    // Warps 9-15, while MMA7 runs: the gated norm of chunk m's tokens
    // kEpiTokens .. 63 (the epilogue takes the others), from the epilogue's
    // staging, over 14 half-warps; the z rows of chunk m+1 are requested once
    // both parts have read chunk m's.
    auto help_norm = [&](int m) {
      const int hw = 2 * (warp - 9) + (lane >> 4);
      __syncwarp();
      bool hok = bar_wait(&V.bar_ofree, (uint32_t)m & 1u);
      hok = bar_wait(&V.bar_z, (uint32_t)m & 1u) && hok;
      const int nv = min(kC, T - kC * m);
      NormRegs<kHelpNR> R;
      norm_load<kHelpNR>(sm, R, nv, kEpiTokens + hw, 14, lane);
      named_sync(kBarHelp, kHelpThreads);
      if (tid == kHelpLeadTid) {
        if (m + 1 < nch) {
          hok = count_wait(&V.epi_zread, m + 1) && hok;
          load_z(m + 1);
        }
        __threadfence_block();
        *reinterpret_cast<volatile int *>(&V.help_loaded) = m + 1;
      }
      if (__all_sync(0xffffffffu, hok && ok))
        norm_store<kHelpNR>(R, static_cast<const bf16 *>(a.norm_w), static_cast<bf16 *>(a.o), d, bos, h, kC * m, nv,
                            kEpiTokens + hw, 14, lane, o_size, a.err);
      ok = ok && hok;
    };
    bool finished = true;
    for (int n = 0; n < nch; ++n) {
      const int st = n & 1;
      const uint32_t sb = sbase + st * kStage;
      // MMA4 D = S (-W^T) (warp 8) once the chunk's tiles are in;
      // MMA5 O1 = S Q^T right after it if the epilogue has read the previous
      // chunk's O1, O2 by then, else after the Delta pass, before MMA7 (so
      // that MMA7's barrier covers MMA5's reads of the fp16 state).  The other
      // chain warps go on to wait for D.  A wait that times out is voted on
      // once, at the chunk's closing barrier.
      __syncwarp();
      const bool w = bar_wait(&V.full[st], (uint32_t)(n >> 1) & 1u);
      ok = ok && w;
      bool o1_done = false;
      auto mma5 = [&]() {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ta_w(tmem + TS_O1, tmem + TS_S16 + 8 * ks, desc_k(sb + Q_Q, ks, kC), id_kk, ks > 0);
      };
      if (issuer && __all_sync(0xffffffffu, w)) {
        fence_after();
        const uint64_t dnw = desc_mn(sb + Q_NW, 0, kD);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_ta_w(tmem + TS_D, tmem + TS_S16 + 8 * ks, dnw + (uint64_t)(ks * 128), id_km, ks > 0);
        commit_w(&V.bar_d);
        o1_done = __all_sync(0xffffffffu, n == 0 || bar_test_wait(&V.bar_ofree, (uint32_t)(n - 1) & 1u));
        if (o1_done) {
          fence_after();
          mma5();
        }
      }
      // Delta^T = D + U^T -> fp16 hi (MMA6) and (Delta Gamma)^T hi / lo (MMA7),
      // once D and U^T are in
      __syncwarp();
      ok = bar_wait(&V.bar_d, (uint32_t)n & 1u) && ok;
      ok = bar_wait(&V.bar_u, (uint32_t)n & 1u) && ok;
      fence_after();
      {
        // this thread: row lrow, token columns 32 ch .. 32 ch + 31 (U^T box ch)
        const float *gam = vec_d(st) + kC + 32 * ch;
        const uint8_t *ub = sm + S_U + ch * 16384 + lrow * 128;
        uint32_t rr[32];
        tmem_ld32_nw(tl + TS_D + 32 * ch, rr);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 u4 = *reinterpret_cast<const float4 *>(ub + ((q ^ (lrow & 7)) << 4));
          rr[4 * q] = __float_as_uint(__uint_as_float(rr[4 * q]) + u4.x);
          rr[4 * q + 1] = __float_as_uint(__uint_as_float(rr[4 * q + 1]) + u4.y);
          rr[4 * q + 2] = __float_as_uint(__uint_as_float(rr[4 * q + 2]) + u4.z);
          rr[4 * q + 3] = __float_as_uint(__uint_as_float(rr[4 * q + 3]) + u4.w);
        }
        {
          uint32_t wh[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) wh[q] = pack2_inrange(__uint_as_float(rr[2 * q]), __uint_as_float(rr[2 * q + 1]));
          tmem_st16w_nw(tl + TS_DH + 16 * ch, wh);
        }
        uint32_t gh[16], gl[16];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {  // times e^{G_last - G_j} <= 1
          const float4 g = ld4(gam + q);
          const float2 p01 = __fmul2_rn(make_float2(__uint_as_float(rr[q]), __uint_as_float(rr[q + 1])), make_float2(g.x, g.y));
          const float2 p23 =
              __fmul2_rn(make_float2(__uint_as_float(rr[q + 2]), __uint_as_float(rr[q + 3])), make_float2(g.z, g.w));
          split2_inrange(p01.x, p01.y, gh[q / 2], gl[q / 2]);
          split2_inrange(p23.x, p23.y, gh[q / 2 + 1], gl[q / 2 + 1]);
        }
        tmem_st16w_nw(tl + TS_DG + 16 * ch, gh);
        tmem_st16w_nw(tl + TS_DG + 32 + 16 * ch, gl);
        tmem_wait_st();
      }
      fence_before();
      named_sync(kBarChain, kChainThreads);
      // U^T is read (the producer may load the next); the deferred MMA5,
      // MMA7 (the state update, first: the chain waits for it), MMA6 (issuer).
      if (issuer) {
        if (lane == 0) mbar_arrive(&V.bar_ufree);
        __syncwarp();
        if (!o1_done) {
          ok = bar_wait(&V.bar_ofree, (uint32_t)(n - 1) & 1u) && ok;
          fence_after();
          mma5();
        }
        fence_after();
        const uint64_t dkh = desc(sb + Q_KH, 8192, 1024), dkl = desc(sb + Q_KL, 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_ta_w(tmem + TS_S, tmem + TS_DG + 8 * ks, dkh + (uint64_t)(ks * 128), id_km128, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_ta_w(tmem + TS_S, tmem + TS_DG + 8 * ks, dkl + (uint64_t)(ks * 128), id_km128, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ta_w(tmem + TS_S, tmem + TS_DG + 32 + 8 * ks, dkh + (uint64_t)(ks * 128), id_km128, 1);
        commit_w(&V.bar_s);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ta_w(tmem + TS_O2, tmem + TS_DH + 8 * ks, desc_k(sb + Q_M, ks, kC), id_kk, ks > 0);
        commit_w(&V.bar_o);
      } else if (n > 0) {
        help_norm(n - 1);
      }
      // The state pass: the fp16 copy and the rescale by the next chunk's
      // decay, or S_T after the last chunk.
      const bool last = n + 1 == nch;
      const float dcn = last ? 1.f : dc_of(n + 1);
      __syncwarp();
      ok = bar_wait(&V.bar_s, (uint32_t)n & 1u) && ok;
      if (tid == kIssuerTid) *reinterpret_cast<volatile int *>(&V.s_seen) = n + 1;
      fence_after();
      {
        uint32_t ra[32];
        auto block = [&](uint32_t(&r0)[32], const int k0) {
          if (last) {
            float4 *dst = reinterpret_cast<float4 *>(a.S_T + unit_off + (long long)lrow * kD + k0);
            if (ok && in_bounds(unit_off + (long long)lrow * kD + k0 + 32, S_size, a.err))
#pragma unroll
              for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1]),
                                     __uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3]));
          } else {
            uint32_t w16[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) w16[q] = pack2_inrange(__uint_as_float(r0[2 * q]), __uint_as_float(r0[2 * q + 1]));
            tmem_st16w_nw(tl + TS_S16 + k0 / 2, w16);
#pragma unroll
            for (int q = 0; q < 32; q += 2) {
              const float2 x0 =
                  __fmul2_rn(make_float2(__uint_as_float(r0[q]), __uint_as_float(r0[q + 1])), make_float2(dcn, dcn));
              r0[q] = __float_as_uint(x0.x);
              r0[q + 1] = __float_as_uint(x0.y);
            }
            tmem_st32w_nw(tl + TS_S + k0, r0);
          }
        };
        const int k0 = 64 * ch;  // this thread's 64 columns
        tmem_ld32_nw(tl + TS_S + k0, ra);
        tmem_wait_ld();
        block(ra, k0);
        tmem_ld32_nw(tl + TS_S + k0 + 32, ra);
        tmem_wait_ld();
        block(ra, k0 + 32);
      }
      tmem_wait_st();
      fence_before();
      // A timeout here or an abort elsewhere ends the loop for all chain warps
      // at once (a warp leaving alone would strand the others at a barrier).
      if (named_sync_or(kBarChain, kChainThreads, !ok || seq_aborted(V))) {
        finished = false;
        break;
      }
    }
    if (finished && !issuer) help_norm(nch - 1);
    if (!ok && (tid == kIssuerTid || tid == kHelpLeadTid)) seq_fail(V, a.err);
  } else {
    // ------------------------------------------- the epilogue (warps 0-6)
    // O staging: warp w takes lane quadrant w & 3, column half w >> 2; lane
    // quadrant 3 has one epilogue warp (3), which takes both halves.  The
    // chunk's d values are copied out first, so that the stage buffer is
    // free for the next load once MMA6 is done (V.epi_seen).
    const int quad = warp & 3;
    const int lrow = 32 * quad + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * quad) << 16);
    const int h_lo = warp < 4 ? 0 : 1, h_hi = warp < 3 ? 1 : 2;
    bool ok = true;
    if (tid == 0) load_z(0);
    for (int n = 0; n < nch; ++n) {
      const int st = n & 1;
      __syncwarp();
      ok = bar_wait(&V.bar_o, (uint32_t)n & 1u) && ok;
      ok = bar_wait(&V.full[st], (uint32_t)(n >> 1) & 1u) && ok;  // this stage's vectors (long landed)
      fence_after();
      if (tid < kC) V.de[n & 1][tid] = vec_d(st)[tid];
      // The chain warps have read chunk n-1's staging (its tokens kEpiTokens..63).
      if (n > 0) ok = count_wait(&V.help_loaded, n) && ok;
      named_sync(kBarEpi, kEpiThreads);
      if (tid == 0) *reinterpret_cast<volatile int *>(&V.epi_seen) = n + 1;  // MMA6 done, the vectors read
      for (int half = h_lo; half < h_hi; ++half) {  // O^T = d (S Q^T) + Delta^T M^T -> staging [i][v]
        float *ost = reinterpret_cast<float *>(sm + S_OST);
        const float *dq = V.de[n & 1] + 32 * half;
#pragma unroll
        for (int c0 = 0; c0 < 32; c0 += 16) {
          uint32_t ra[16], rb[16];
          tmem_ld16_nw(tl + TS_O1 + 32 * half + c0, ra);
          tmem_ld16_nw(tl + TS_O2 + 32 * half + c0, rb);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 16; q += 4) {
            const float4 dd = ld4(dq + c0 + q);
            const float2 o01 = __ffma2_rn(make_float2(dd.x, dd.y), make_float2(__uint_as_float(ra[q]), __uint_as_float(ra[q + 1])),
                                          make_float2(__uint_as_float(rb[q]), __uint_as_float(rb[q + 1])));
            const float2 o23 = __ffma2_rn(make_float2(dd.z, dd.w),
                                          make_float2(__uint_as_float(ra[q + 2]), __uint_as_float(ra[q + 3])),
                                          make_float2(__uint_as_float(rb[q + 2]), __uint_as_float(rb[q + 3])));
            ost[(32 * half + c0 + q + 0) * kD + lrow] = o01.x;
            ost[(32 * half + c0 + q + 1) * kD + lrow] = o01.y;
            ost[(32 * half + c0 + q + 2) * kD + lrow] = o23.x;
            ost[(32 * half + c0 + q + 3) * kD + lrow] = o23.y;
          }
        }
      }
      fence_before();
      named_sync(kBarEpi, kEpiThreads);
      if (tid == 0) mbar_arrive(&V.bar_ofree);  // O1 and O2 are read: MMA5, MMA6 of the next chunk may write them
      // The gated norm of the chunk's tokens 0 .. kEpiTokens-1 over 14
      // half-warps (the chain warps take the rest during the next chunk's
      // MMA7): staged O and z into registers, then y formed and stored.
      __syncwarp();
      ok = bar_wait(&V.bar_z, (uint32_t)n & 1u) && ok;
      const int nv = min(kC, T - kC * n), nv0 = min(nv, kEpiTokens), i0 = 2 * warp + (lane >> 4);
      NormRegs<kEpiNR> R;
      norm_load<kEpiNR>(sm, R, nv0, i0, 14, lane);
      named_sync(kBarEpi, kEpiThreads);
      if (tid == 0) {  // this role's z rows are in registers (the chain warps reload z)
        __threadfence_block();
        *reinterpret_cast<volatile int *>(&V.epi_zread) = n + 1;
      }
      if (__all_sync(0xffffffffu, ok))  // warp-uniform: the norm's shuffles need the whole warp
        norm_store<kEpiNR>(R, static_cast<const bf16 *>(a.norm_w), static_cast<bf16 *>(a.o), d, bos, h, kC * n, nv0, i0,
                           14, lane, o_size, a.err);
      // The staging is read; a timeout here or an abort elsewhere ends the
      // loop for all epilogue warps at once.
      if (named_sync_or(kBarEpi, kEpiThreads, !ok || seq_aborted(V))) break;
    }
    if (!ok && tid == 0) seq_fail(V, a.err);
  }

  write_conv_T();
  // Before the CTA ends: no copy still landing in shared memory and no MMA
  // still writing TMEM (after an early exit; on a normal exit every request
  // was consumed and every MMA waited for).
  fence_before();
  __syncthreads();
  if (tid == kIssuerTid) {
    for (int st = 0; st < 2; ++st)
      if (V.req_full[st] > 0) bar_wait(&V.full[st], (uint32_t)(V.req_full[st] - 1) & 1u);
    if (V.req_u > 0) bar_wait(&V.bar_u, (uint32_t)(V.req_u - 1) & 1u);
    if (V.req_z > 0) bar_wait(&V.bar_z, (uint32_t)(V.req_z - 1) & 1u);
    commit(&V.bar_end);
    bar_wait(&V.bar_end, 0);
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kSeqTmem);
  }
}

__global__ void __launch_bounds__(kSeqThreads, 1)
    prefill_seq_kernel(const PrefillArgs a, const SplitArgs s, const __grid_constant__ CUtensorMap tm_qk,
                       const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_u,
                       const __grid_constant__ CUtensorMap tm_nw, const __grid_constant__ CUtensorMap tm_m) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  seq_role(a, s, &tm_qk, &tm_z, &tm_u, &tm_nw, &tm_m, sm, nullptr);
}

// =============================================================================
// prefill_overlap_kernel
// =============================================================================
// Both parts in one cooperative launch, for a fixed-length batch with few
// (sequence, value head) units: CTAs 0 .. B*Hv - 1 run the sequential part,
// every other CTA runs two prep groups, which walk the items chunk by chunk
// and flag each item once its outputs have landed; a sequential CTA reads a
// chunk's outputs once its flag is set.  Every CTA is resident at once (the
// launch is cooperative) and the prep groups wait on nothing the sequential
// CTAs do, so each flag wait ends; a wait that runs past its bound reports
// GDN_ERR_TIMEOUT instead.
constexpr uint32_t kPrepGroupBytes = ((P_VEC + (uint32_t)sizeof(PrepShared) + 1023) / 1024) * 1024;
constexpr uint32_t kOverlapSmem = kSeqSmem > 2 * kPrepGroupBytes + 1024 ? kSeqSmem : 2 * kPrepGroupBytes + 1024;
static_assert(kSeqThreads == 2 * kPrepThreads && kOverlapSmem <= 232448, "two prep groups in a sequential CTA's place");

template <bool kRawGates>
__global__ void __launch_bounds__(kSeqThreads, 1)
    prefill_overlap_kernel(const PrefillArgs a, const SplitArgs s, int *flags,
                           const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_qk,
                           const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_u,
                           const __grid_constant__ CUtensorMap tm_nw, const __grid_constant__ CUtensorMap tm_m) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int nseq = a.d.B * a.d.Hv;
  if ((int)blockIdx.x < nseq) {
    seq_role(a, s, &tm_qk, &tm_z, &tm_u, &tm_nw, &tm_m, sm, flags);
    return;
  }
  PrepShared &V0 = *reinterpret_cast<PrepShared *>(sm + P_VEC);
  if (threadIdx.x < 32) tmem_alloc(&V0.tmem, 2 * kPrepTmem);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = V0.tmem;
  const int g = (int)threadIdx.x / kPrepThreads;
  const PrepGroup G{sm + g * kPrepGroupBytes,
                    tmem + (uint32_t)(g * kPrepTmem),
                    (int)threadIdx.x % kPrepThreads,
                    kBarPrep + 2 * g,
                    kBarSolve + 2 * g,
                    2LL * ((int)blockIdx.x - nseq) + g,
                    2LL * ((int)gridDim.x - nseq),
                    flags};
  prep_role<kRawGates>(a, s, &tm_qkv, &tm_qk, &tm_u, &tm_nw, &tm_m, G);
  fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    fence_after();
    tmem_dealloc(tmem, 2 * kPrepTmem);
  }
}

// ---- tensor maps -------------------------------------------------------------
bool encode_2d(CUtensorMap *m, void *base, CUtensorMapDataType dt, int esize, long long inner, long long rows,
               int box_inner, int box_rows, CUtensorMapSwizzle sw) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(inner * esize)};
  const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// A token-major [rows][width] bf16 tensor with boxes of 128 columns x box_rows rows.
bool encode_rows(CUtensorMap *m, const void *base, long long width, long long rows, int box_rows) {
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
// The staged q^ / k^ [3][rows][Hk*128] fp16 with 128-byte-swizzled 64 x 64 boxes.
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

struct SplitMaps {
  CUtensorMap u, nw, m;
};
bool encode_split(SplitMaps *mp, const SplitArgs &s, long long nitems) {
  return encode_2d(&mp->u, s.ws_u, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2 * 32, nitems * kD, 32, kD,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_2d(&mp->nw, s.ws_nw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, 64, nitems * kD, 64, kD,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_2d(&mp->m, s.ws_m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, 64, nitems * kC, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

long long split_items(const Dims &d, long long tokens, bool packed, int *nslots, int *nch) {
  const long long T = d.T;
  const long long ch = (T + kC - 1) / kC;
  const long long slots = packed ? (tokens >> 6) + d.B + 2 : (long long)d.B * ch;
  *nch = (int)ch;
  *nslots = (int)slots;
  return slots * d.Hv;
}

cudaError_t launch_prefill_split(const PrefillArgs &a, const SplitArgs &s, cudaStream_t st) {
  if (!a.qk_ws || !a.conv_w) return cudaErrorInvalidValue;
  const long long rows = a.cu_seqlens ? (long long)a.d.T : (long long)a.d.B * a.d.T;
  const long long nitems = (long long)s.nslots * a.d.Hv;
  if (nitems * kD >= (1LL << 31) || rows > 0x7fffffffLL - 2 * kC) return cudaErrorInvalidValue;
  CUtensorMap tm_qkv, tm_z, tm_qk;
  SplitMaps mp;
  if (!encode_rows(&tm_qkv, a.qkv_pre, a.d.C, rows, kRawRows) ||
      !encode_rows(&tm_z, a.z, (long long)a.d.Hv * kD, rows, kC) || !encode_qk(&tm_qk, a.qk_ws, a.d.Hk, rows) ||
      !encode_split(&mp, s, nitems))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0, coop = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return e;
  const bool raw = a.gate.g == nullptr;
  // Few units of a fixed-length batch: both parts in one launch, the prep
  // groups on the SMs the sequential CTAs leave (at least half of them).
  const long long nseq = (long long)a.d.B * a.d.Hv;
  if (!s.cu && s.flags && coop && 2 * nseq <= sms) {
    auto ov = raw ? prefill_overlap_kernel<true> : prefill_overlap_kernel<false>;
    e = cudaFuncSetAttribute(ov, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOverlapSmem);
    int per_sm = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ov, kSeqThreads, kOverlapSmem);
    if (e != cudaSuccess) return e;
    if (per_sm >= 1) {
      cudaLaunchConfig_t cfg{};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.gridDim = dim3((unsigned)sms);
      cfg.blockDim = dim3(kSeqThreads);
      cfg.dynamicSmemBytes = kOverlapSmem;
      cfg.stream = st;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, ov, a, s, s.flags, tm_qkv, tm_qk, tm_z, mp.u, mp.nw, mp.m);
    }
  }
  auto prep = raw ? prefill_prep_kernel<true> : prefill_prep_kernel<false>;
  e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
  if (e != cudaSuccess) return e;
  long long grid = 2LL * sms;
  if (grid > nitems) grid = nitems;
  if (grid < 1) grid = 1;
  prep<<<(unsigned)grid, kPrepThreads, kPrepSmem, st>>>(a, s, tm_qkv, tm_qk, mp.u, mp.nw, mp.m);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSeqSmem);
  if (e != cudaSuccess) return e;
  prefill_seq_kernel<<<(unsigned)(a.d.B * a.d.Hv), kSeqThreads, kSeqSmem, st>>>(a, s, tm_qk, tm_z, mp.u, mp.nw, mp.m);
  return cudaGetLastError();
}

}  // namespace gdn
