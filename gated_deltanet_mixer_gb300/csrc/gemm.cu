// gemm.cu -- the projections around the mixer: y[t, n] = sum_k x[t, k] w[n, k]
// (nodes gdn.in_proj, K=5120 -> N=16480, and gdn.out_proj, K=6144 -> N=5120,
// of the page "Qwen3.8-27B"), bf16 in and out, fp32 accumulation, on the
// tcgen05 tensor cores.
//
// A persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: 128 x 64 tiles of x and 256 x 64 tiles of w into a
//               4-stage ring of 128-byte-swizzled shared memory
//   warp 1      MMA issuer: per stage four 128 x 256 x 16 MMAs into one of two
//               TMEM accumulators (2 x 256 fp32 columns); commits free the stage
//               and, after the last k step, hand the tile to the epilogue
//   warps 2-5   epilogue: TMEM -> registers -> bf16, each column range to its
//               output tensor (the in_proj output goes straight into the mixer's
//               qkv_pre | z | b | a buffers), while the MMAs of the next tile run
//               in the other accumulator
// Every wait is an mbarrier wait bounded by the global timer; a timeout sets
// the device error word and the roles leave their loops.
#include <cuda.h>
#include <cuda_bf16.h>

#include "launch.h"
#include "tma_host.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr uint32_t kStageA = BM * BK * 2;                // 16 KB
constexpr uint32_t kStageB = BN * BK * 2;                // 32 KB
constexpr uint32_t kStageBytes = kStageA + kStageB;      // 48 KB
constexpr uint32_t kBarOff = kStages * kStageBytes;      // 192 KB
constexpr uint32_t kSmem = kBarOff + 256 + 1024;         // + barriers + alignment slack
constexpr int kThreads = 192;
static_assert(kSmem <= 232448, "shared memory per CTA");

// Instruction descriptor, kind::f16 with bf16 A and B (format 1), fp32 D.
constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[2], tempty[2];
  uint64_t end;
  uint32_t tmem;
};

// Tile t of the persistent schedule -> (m tile, n tile).  Bands of 8 m tiles
// walk across n, so the CTAs running at once share their w tiles in L2.
__device__ __forceinline__ void tile_of(int t, int tiles_m, int tiles_n, int &mt, int &nt) {
  constexpr int G = 8;
  const int band = t / (G * tiles_n), r = t % (G * tiles_n);
  const int rows = min(G, tiles_m - band * G);
  mt = band * G + r % rows;
  nt = r / rows;
}

__device__ __forceinline__ void store_bf16x8(__nv_bfloat16 *p, const float *v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&t);
  }
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const GemmArgs g, const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  Bars &B = *reinterpret_cast<Bars *>(sm + kBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tiles_m = (g.M + BM - 1) / BM, tiles_n = (g.N + BN - 1) / BN;
  const int ntiles = tiles_m * tiles_n;
  const int nk = (g.K + BK - 1) / BK;
  const uint32_t sbase = smem_u32(sm);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      bar_init(&B.full[s], 1);
      bar_init(&B.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      bar_init(&B.tfull[a], 1);
      bar_init(&B.tempty[a], 4);
    }
    bar_init(&B.end, 1);
  }
  if (warp == 1) tmem_alloc(&B.tmem, 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = B.tmem;
  bool ok = true;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        int mt, nt;
        tile_of(t, tiles_m, tiles_n, mt, nt);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (!bar_wait(&B.empty[s], ((it / kStages) & 1) ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + s * kStageBytes;
          bar_expect_tx(&B.full[s], kStageBytes);
          tma_load_3d(dst, &tm_x, kb * BK, mt * BM, 0, &B.full[s]);
          tma_load_3d(dst + kStageA, &tm_w, kb * BK, nt * BN, 0, &B.full[s]);
        }
      }
      // Leave only when every stage issued has been consumed (bounded).
      if (ok && it > 0)
        for (uint32_t j = (it > kStages ? it - kStages : 0); j < it; ++j)
          if (!bar_wait(&B.empty[j % kStages], (j / kStages) & 1)) {
            ok = false;
            break;
          }
      if (!ok) atomicOr(g.err, kErrTimeout);
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t id = idesc_bf16(BM, BN);
      uint32_t it = 0;
      int local = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++local) {
        const int acc = local & 1;
        if (!bar_wait(&B.tempty[acc], ((local >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (!bar_wait(&B.full[s], (it / kStages) & 1)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t a0 = sbase + s * kStageBytes, b0 = a0 + kStageA;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            mma(d, desc_k(a0, ks, BM), desc_k(b0, ks, BN), id, (kb > 0 || ks > 0) ? 1u : 0u);
          commit(&B.empty[s]);
        }
        if (!ok) break;
        commit(&B.tfull[acc]);
      }
      commit(&B.end);  // every MMA issued is complete before TMEM is freed
      if (!bar_wait(&B.end, 0)) ok = false;
      if (!ok) atomicOr(g.err, kErrTimeout);
    }
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = tile rows
    const int quad = warp & 3;
    const int r_in = 32 * quad + lane;
    int local = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++local) {
      int mt, nt;
      tile_of(t, tiles_m, tiles_n, mt, nt);
      const int acc = local & 1;
      const bool got = bar_wait(&B.tfull[acc], (local >> 1) & 1);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) atomicOr(g.err, kErrTimeout);
        break;
      }
      fence_after();
      const long long row = (long long)mt * BM + r_in;
      const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld32(taddr + c, v);  // every lane of the warp takes part
        const int col0 = nt * BN + c;
        if (row >= g.M || col0 >= g.N) continue;
        for (int o = 0; o < g.n_out; ++o) {
          const GemmOut &out = g.out[o];
          const int lo = max(col0, out.col_begin), hi = min(min(col0 + 32, out.col_end), g.N);
          if (lo >= hi) continue;
          __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(out.ptr) + row * out.ld - out.col_begin;
          if (lo == col0 && hi == col0 + 32 && out.vec_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q) store_bf16x8(dst + col0 + 8 * q, v + 8 * q);
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if (col0 + q >= lo && col0 + q < hi) dst[col0 + q] = __float2bfloat16_rn(v[q]);
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) {  // this warp has read its lanes: the accumulator may be refilled
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&B.tempty[acc])) : "memory");
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// A row-major [rows][K] bf16 matrix as a 3-d map (third extent 1) with
// 128-byte-swizzled boxes of 64 columns x box_rows rows.
bool encode_kmajor(CUtensorMap *m, const void *base, long long rows, long long K, long long ld, int box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, 1};
  const cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * rows};
  const cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs &a, int num_sms, cudaStream_t s) {
  CUtensorMap tm_x, tm_w;
  if (!encode_kmajor(&tm_x, a.x, a.M, a.K, a.ldx, BM) || !encode_kmajor(&tm_w, a.w, a.N, a.K, a.ldw, BN))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  const long long ntiles = (long long)((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = (int)(ntiles < num_sms ? ntiles : num_sms);
  gemm_kernel<<<grid, kThreads, kSmem, s>>>(a, tm_x, tm_w);
  return cudaGetLastError();
}

}  // namespace gdn
