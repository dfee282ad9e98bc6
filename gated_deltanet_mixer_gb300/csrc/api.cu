// api.cu -- the C ABI of libgdn (declared in include/gdn.h): argument checks,
// aliasing rules, and the launch of the kernels on the caller's stream.
#include <cmath>
#include <cstdint>

#include "gdn.h"
#include "launch.h"

namespace {

// One error word per device that loads the library: kernels OR bits into it.
__device__ unsigned int g_err_word;

struct Range {
  uintptr_t lo, hi;  // [lo, hi); empty when lo == hi
};

Range range_of(const void *p, size_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + (p ? bytes : 0)};
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Sizes {
  size_t io;     // bytes per io element
  size_t qkv, zo, gb, S, conv, conv_w, norm_w;  // bytes of each tensor
};

gdn_status check_shape(const gdn_shape *sh, bool decode, gdn::Dims *d, Sizes *z) {
  if (!sh) return GDN_ERR_INVALID_ARG;
  if (sh->B < 1 || sh->T < 1 || sh->Hk < 1 || sh->Hv < 1 || sh->Dk < 1 || sh->Dv < 1)
    return GDN_ERR_INVALID_ARG;
  if (decode && sh->T != 1) return GDN_ERR_INVALID_ARG;
  if (sh->io_dtype != GDN_F32 && sh->io_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (!std::isfinite(sh->eps_l2) || sh->eps_l2 < 0.f || !std::isfinite(sh->eps_norm) ||
      sh->eps_norm < 0.f || !std::isfinite(sh->q_scale))
    return GDN_ERR_INVALID_ARG;
  if (sh->Dk != gdn::kDHead || sh->Dv != gdn::kDHead) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (sh->Hv % sh->Hk != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
  // Limits that keep every size product inside 64 bits and the grid legal.
  if (sh->Hk > 4096 || sh->Hv > 4096 || sh->B > 65536 || (long long)sh->B * sh->T > (1LL << 34))
    return GDN_ERR_UNSUPPORTED_SHAPE;
  d->B = sh->B;
  d->T = sh->T;
  d->Hk = sh->Hk;
  d->Hv = sh->Hv;
  d->C = 2LL * sh->Hk * gdn::kDHead + (long long)sh->Hv * gdn::kDHead;
  d->eps_l2 = sh->eps_l2;
  d->eps_norm = sh->eps_norm;
  d->q_scale = sh->q_scale != 0.f ? sh->q_scale : 1.0f / std::sqrt((float)gdn::kDHead);
  const size_t BT = (size_t)sh->B * sh->T;
  z->io = sh->io_dtype == GDN_BF16 ? 2 : 4;
  z->qkv = BT * (size_t)d->C * z->io;
  z->zo = BT * (size_t)sh->Hv * gdn::kDHead * z->io;
  z->gb = BT * (size_t)sh->Hv * sizeof(float);
  z->S = (size_t)sh->B * sh->Hv * gdn::kDHead * gdn::kDHead * sizeof(float);
  z->conv = (size_t)sh->B * 3 * (size_t)d->C * z->io;
  z->conv_w = (size_t)d->C * 4 * z->io;
  z->norm_w = (size_t)gdn::kDHead * z->io;
  return GDN_OK;
}

gdn_status check_device(unsigned int **err) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (major != 10 || minor != 3) return GDN_ERR_NO_DEVICE;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(err), g_err_word) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char *gdn_status_str(int s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument";
    case GDN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case GDN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case GDN_ERR_ALIAS: return "forbidden buffer overlap";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_TIMEOUT: return "device-side wait timed out";
    case GDN_ERR_NO_DEVICE: return "current device is not an sm_103 GPU";
    default: return "unknown status";
  }
}

gdn_status gdn_prefill(const gdn_shape *shape, const void *qkv_pre, const void *z,
                       const float *g, const float *beta, const void *conv_w,
                       const void *norm_w, const float *S0, const void *conv0, void *o,
                       float *S_T, void *conv_T, void *stream) {
  gdn::Dims d;
  Sizes sz;
  gdn_status st = check_shape(shape, false, &d, &sz);
  if (st != GDN_OK) return st;
  if (!qkv_pre || !z || !g || !beta || !conv_w || !norm_w || !o || !S_T || !conv_T)
    return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {qkv_pre, z, g, beta, conv_w, norm_w, S0, conv0, o, S_T, conv_T};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
  const Range in[] = {range_of(qkv_pre, sz.qkv), range_of(z, sz.zo),   range_of(g, sz.gb),
                      range_of(beta, sz.gb),     range_of(conv_w, sz.conv_w),
                      range_of(norm_w, sz.norm_w), range_of(S0, sz.S), range_of(conv0, sz.conv)};
  const Range ro = range_of(o, sz.zo), rs = range_of(S_T, sz.S), rc = range_of(conv_T, sz.conv);
  const bool in_place = S0 != nullptr && S0 == S_T;
  for (int i = 0; i < 8; ++i) {
    if (overlap(ro, in[i]) || overlap(rc, in[i])) return GDN_ERR_ALIAS;
    if (i == 6 && in_place) continue;
    if (overlap(rs, in[i])) return GDN_ERR_ALIAS;
  }
  if (overlap(ro, rs) || overlap(ro, rc) || overlap(rs, rc)) return GDN_ERR_ALIAS;
  unsigned int *err = nullptr;
  st = check_device(&err);
  if (st != GDN_OK) return st;

  gdn::PrefillArgs a{d, qkv_pre, z, g, beta, conv_w, norm_w, S0, conv0, o, S_T, conv_T, err};
  // bf16 io: the chunked tensor-core kernel; fp32 io: the exact token-serial kernel.
  const bool bf16 = shape->io_dtype == GDN_BF16;
  cudaError_t e = bf16 ? gdn::launch_prefill_chunked(a, true, (cudaStream_t)stream)
                       : gdn::launch_prefill(a, false, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_decode_step(const gdn_shape *shape, const void *qkv_pre, const void *z,
                           const float *g, const float *beta, const void *conv_w,
                           const void *norm_w, float *S, const void *conv_in, void *conv_out,
                           void *o, void *stream) {
  gdn::Dims d;
  Sizes sz;
  gdn_status st = check_shape(shape, true, &d, &sz);
  if (st != GDN_OK) return st;
  if (!qkv_pre || !z || !g || !beta || !conv_w || !norm_w || !S || !conv_in || !conv_out || !o)
    return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {qkv_pre, z, g, beta, conv_w, norm_w, S, conv_in, conv_out, o};
  for (const void *p : ptrs)
    if (!aligned16(p)) return GDN_ERR_ALIGNMENT;
  const Range in[] = {range_of(qkv_pre, sz.qkv), range_of(z, sz.zo), range_of(g, sz.gb),
                      range_of(beta, sz.gb),     range_of(conv_w, sz.conv_w),
                      range_of(norm_w, sz.norm_w), range_of(conv_in, sz.conv)};
  const Range rS = range_of(S, sz.S), ro = range_of(o, sz.zo), rc = range_of(conv_out, sz.conv);
  for (const Range &r : in)
    if (overlap(rS, r) || overlap(ro, r) || overlap(rc, r)) return GDN_ERR_ALIAS;
  if (overlap(rS, ro) || overlap(rS, rc) || overlap(ro, rc)) return GDN_ERR_ALIAS;
  unsigned int *err = nullptr;
  st = check_device(&err);
  if (st != GDN_OK) return st;

  gdn::DecodeArgs a{d, qkv_pre, z, g, beta, conv_w, norm_w, S, conv_in, conv_out, o, err};
  cudaError_t e = gdn::launch_decode(a, shape->io_dtype == GDN_BF16, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_device_status(void *stream, int reset) {
  cudaStream_t s = (cudaStream_t)stream;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbolAsync(&word, g_err_word, sizeof(word), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (reset) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_err_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return GDN_ERR_CUDA;
  }
  return (word & gdn::kErrTimeout) ? GDN_ERR_TIMEOUT : GDN_OK;
}

}  // extern "C"
