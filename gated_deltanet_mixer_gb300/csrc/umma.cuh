// umma.cuh -- inline-PTX wrappers for the sm_100-family tensor-core path:
// tcgen05.mma (fp16 operands, fp32 accumulate in TMEM), TMEM alloc / ld / st,
// mbarriers with bounded waits, and the shared-memory operand layouts.
//
// Operand tiles use the 128-byte swizzle: an "atom" is 8 rows of 128 bytes
// (64 16-bit values) = 1024 bytes, 16-byte chunk c of row r stored at chunk c ^ (r % 8).
// K-major: rows are the M (or N) index, the contraction index contiguous;
//   a tile of R rows keeps K in blocks of 64 (R * 128 bytes each), 8-row
//   groups 1024 bytes apart (SBO); one K step of 16 advances 32 bytes.
// MN-major: rows are the contraction index, the M (or N) index contiguous;
//   M/N in blocks of 64 (LBO apart), 8-row K groups 1024 bytes apart (SBO);
//   one K step of 16 advances 2048 bytes.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace gdn {
namespace umma {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Byte offset of element (r, k) in a K-major tile of R rows.
__device__ __forceinline__ uint32_t kmaj(int r, int k, int R) {
  return (uint32_t)((k >> 6) * (R * 128) + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}
// Byte offset of element (mn, k) in an MN-major tile whose contraction extent is Kdim.
__device__ __forceinline__ uint32_t mnmaj(int mn, int k, int Kdim) {
  return (uint32_t)((mn >> 6) * ((Kdim >> 3) * 1024) + (k >> 3) * 1024 + (k & 7) * 128 +
                    ((((mn & 63) >> 3) ^ (k & 7)) << 4) + (mn & 7) * 2);
}

// Shared-memory matrix descriptor (version 1, 128-byte swizzle).
__device__ __forceinline__ uint64_t desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// K step `ks` (16 elements) of a K-major tile of R rows.
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int ks, int R) {
  return desc(base + (uint32_t)((ks >> 2) * (R * 128) + (ks & 3) * 32), 16, 1024);
}
// K step `ks` of an MN-major tile whose contraction extent is Kdim.
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int ks, int Kdim) {
  return desc(base + (uint32_t)(ks * 2048), (uint32_t)((Kdim >> 3) * 1024), 1024);
}

// Instruction descriptor, kind::f16: fp16 A and B (format 0), fp32 D (format 1).
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
// The same with A read from TMEM: lane m holds row m, 32-bit column c holds
// the fp16 pair (2c, 2c+1) along K, so one K step of 16 advances 8 columns.
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate));
}
// The same two, executed by every lane of a converged warp with the same
// operands; lane 0 issues.  The warp stays converged, so the operands need not
// leave a divergent region: about half the issue time of a lone thread.
__device__ __forceinline__ void mma_w(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
__device__ __forceinline__ void mma_ta_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate));
}
// commit() by lane 0 of a converged warp (the lane that issued with mma_w).
__device__ __forceinline__ void commit_w(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(smem_u32(bar))
      : "memory");
}
// Arrive on `bar` once every previously issued MMA of this thread completes.
__device__ __forceinline__ void commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the MMA unit.
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- mbarriers
__device__ __forceinline__ void bar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool bar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for phase `parity`: false if it has not completed within
// `limit_ns` (default about one second; the work it waits for takes
// microseconds).
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity,
                                         uint64_t limit_ns = 1000000000ull) {
  if (bar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!bar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}
// Arrive on `bar` announcing `bytes` of asynchronous copies to complete on it.
__device__ __forceinline__ void bar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Announce `bytes` more of asynchronous copies on `bar` without arriving
// (the phase still waits for its arrival).
__device__ __forceinline__ void bar_expect_tx_only(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// TMA: a 3-d box of a tensor map into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// ---- TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
// 32 consecutive fp32 columns of this warp's 32 lanes (lane = thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// The same without the wait (raw words): several loads in flight, then
// tmem_wait_ld() before any of the registers is used.
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Stores without the wait; tmem_wait_st() before the written columns are
// consumed (by this thread or, after a barrier, by the MMA unit).
__device__ __forceinline__ void tmem_st16w_nw(uint32_t taddr, const uint32_t (&w)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]));
}
__device__ __forceinline__ void tmem_st32w_nw(uint32_t taddr, const uint32_t (&w)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
      "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
      "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31]));
}
// 16 consecutive 32-bit columns (raw words) of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st16w(uint32_t taddr, const uint32_t (&w)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]));
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])));
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// fp16 operand value: round to nearest, clamped to the finite fp16 range.
constexpr float kHalfMax = 65504.0f;
__device__ __forceinline__ __half to_h(float x) {
  return __float2half_rn(fminf(fmaxf(x, -kHalfMax), kHalfMax));
}
// A pair of floats as packed fp16 (a in the low half), rounded to nearest and
// saturated to the finite range (+-65504) in the conversion itself; NaN stays
// NaN.  Finite values inside the range convert exactly as __floats2half2_rn.
__device__ __forceinline__ uint32_t pack2_sat(float a, float b) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));  // first source -> high half
  return r;
}
// Pack 8 floats into one 16-byte chunk of fp16 and store it to shared memory.
__device__ __forceinline__ void st_h8(uint8_t *p, const float *v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 t = __halves2half2(to_h(v[2 * i]), to_h(v[2 * i + 1]));
    w[i] = *reinterpret_cast<uint32_t *>(&t);
  }
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// The same, as a hi/lo pair of fp16 chunks: hi = fp16(v), lo = fp16(v - hi), so
// that hi + lo carries about 22 significant bits into an MMA pair.
__device__ __forceinline__ void st_h8_split(uint8_t *phi, uint8_t *plo, const float *v) {
  uint32_t wh[4], wl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half h0 = to_h(v[2 * i]), h1 = to_h(v[2 * i + 1]);
    const __half l0 = to_h(v[2 * i] - __half2float(h0)), l1 = to_h(v[2 * i + 1] - __half2float(h1));
    __half2 th = __halves2half2(h0, h1), tl = __halves2half2(l0, l1);
    wh[i] = *reinterpret_cast<uint32_t *>(&th);
    wl[i] = *reinterpret_cast<uint32_t *>(&tl);
  }
  *reinterpret_cast<uint4 *>(phi) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
  *reinterpret_cast<uint4 *>(plo) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
}

}  // namespace umma
}  // namespace gdn
