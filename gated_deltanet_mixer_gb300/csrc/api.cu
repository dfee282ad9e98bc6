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
  size_t io;                                                     // bytes per io element
  size_t qkv, zo, gb, gio, S, conv, conv_w, norm_w, head, snap;  // bytes of each tensor
};

// tokens: rows of the token-major tensors (B*T fixed length, T packed).
gdn_status check_shape(const gdn_shape *sh, long long tokens, gdn::Dims *d, Sizes *z) {
  if (!sh) return GDN_ERR_INVALID_ARG;
  if (sh->B < 1 || sh->T < 1 || sh->Hk < 1 || sh->Hv < 1 || sh->Dk < 1 || sh->Dv < 1)
    return GDN_ERR_INVALID_ARG;
  if (sh->io_dtype != GDN_F32 && sh->io_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (!std::isfinite(sh->eps_l2) || sh->eps_l2 < 0.f || !std::isfinite(sh->eps_norm) ||
      sh->eps_norm < 0.f || !std::isfinite(sh->q_scale))
    return GDN_ERR_INVALID_ARG;
  if (sh->Dk != gdn::kDHead || sh->Dv != gdn::kDHead) return GDN_ERR_UNSUPPORTED_SHAPE;
  if (sh->Hv % sh->Hk != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
  // Limits that keep every size product inside 64 bits, the grid legal and
  // token row indices (TMA coordinates) inside 31 bits.
  if (sh->Hk > 4096 || sh->Hv > 4096 || sh->B > 65536 || tokens > (1LL << 30))
    return GDN_ERR_UNSUPPORTED_SHAPE;
  d->B = sh->B;
  d->T = sh->T;
  d->Hk = sh->Hk;
  d->Hv = sh->Hv;
  d->C = 2LL * sh->Hk * gdn::kDHead + (long long)sh->Hv * gdn::kDHead;
  d->eps_l2 = sh->eps_l2;
  d->eps_norm = sh->eps_norm;
  d->q_scale = sh->q_scale != 0.f ? sh->q_scale : 1.0f / std::sqrt((float)gdn::kDHead);
  const size_t N = (size_t)tokens;
  z->io = sh->io_dtype == GDN_BF16 ? 2 : 4;
  z->qkv = N * (size_t)d->C * z->io;
  z->zo = N * (size_t)sh->Hv * gdn::kDHead * z->io;
  z->gb = N * (size_t)sh->Hv * sizeof(float);
  z->gio = N * (size_t)sh->Hv * z->io;
  z->S = (size_t)sh->B * sh->Hv * gdn::kDHead * gdn::kDHead * sizeof(float);
  z->conv = (size_t)sh->B * 3 * (size_t)d->C * z->io;
  z->conv_w = (size_t)d->C * 4 * z->io;
  z->norm_w = (size_t)gdn::kDHead * z->io;
  z->head = (size_t)sh->Hv * sizeof(float);
  z->snap = N * (size_t)sh->Hv * gdn::kDHead * gdn::kDHead * sizeof(float);
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

// The gate source: (g, beta) or the raw projections, never both.
gdn_status gate_source(const float *g, const float *beta, const gdn_raw_gates *raw, gdn::GateSrc *out) {
  if (raw) {
    if (g || beta || !raw->a || !raw->b || !raw->A_log || !raw->dt_bias) return GDN_ERR_INVALID_ARG;
    *out = gdn::GateSrc{nullptr, nullptr, raw->a, raw->b, raw->A_log, raw->dt_bias};
  } else {
    if (!g || !beta) return GDN_ERR_INVALID_ARG;
    *out = gdn::GateSrc{g, beta, nullptr, nullptr, nullptr, nullptr};
  }
  return GDN_OK;
}

// The gate tensors of either source, as input ranges; returns how many.
int gate_ranges(const gdn::GateSrc &gs, const Sizes &sz, Range *out) {
  if (gs.g) {
    out[0] = range_of(gs.g, sz.gb);
    out[1] = range_of(gs.beta, sz.gb);
    return 2;
  }
  out[0] = range_of(gs.a, sz.gio);
  out[1] = range_of(gs.b, sz.gio);
  out[2] = range_of(gs.A_log, sz.head);
  out[3] = range_of(gs.dt_bias, sz.head);
  return 4;
}

bool all_aligned(const void *const *ptrs, int n) {
  for (int i = 0; i < n; ++i)
    if (ptrs[i] && !aligned16(ptrs[i])) return false;
  return true;
}

// Workspace of the staged q^ / k^: 3 fp16 values per (token row, key head, channel).
size_t qk_workspace_bytes(const gdn::Dims &d, long long tokens) {
  return 3 * (size_t)tokens * (size_t)d.Hk * gdn::kDHead * 2;
}
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
// The chunk-parallel form pays where the sequential kernel alone (one CTA per
// sequence and value head, one per SM) cannot fill the GPU twice over: there
// the state-independent work moves onto the idle SMs.  With more units the
// staged form keeps every SM busy and moves fewer bytes.
bool split_pays(long long units) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return true;
  return units < 2LL * sms;
}
// Workspace of the chunk-parallel / sequential prefill: the staged q^ / k^,
// then kSplitItemBytes per (chunk slot, value head); 0 when the work items
// exceed what the kernels index (TMA row coordinates in 31 bits).
size_t split_workspace_bytes(const gdn::Dims &d, long long tokens, bool packed, gdn::SplitArgs *sa = nullptr) {
  int nslots = 0, nch = 0;
  const long long items = gdn::split_items(d, tokens, packed, &nslots, &nch);
  if (items < 1 || items * gdn::kDHead >= (1LL << 31)) return 0;
  if (sa) {
    sa->B = d.B;
    sa->T = d.T;
    sa->nch = nch;
    sa->nslots = nslots;
  }
  return align256(qk_workspace_bytes(d, tokens)) + (size_t)items * gdn::kSplitItemBytes;
}

gdn_status prefill_impl(const gdn_shape *shape, const gdn_prefill_io *io, void *stream) {
  if (!shape || !io) return GDN_ERR_INVALID_ARG;
  if (shape->B < 1 || shape->T < 1) return GDN_ERR_INVALID_ARG;
  const bool packed = io->cu_seqlens != nullptr;
  const long long tokens = packed ? (long long)shape->T : (long long)shape->B * shape->T;
  gdn::Dims d;
  Sizes sz;
  gdn_status st = check_shape(shape, tokens, &d, &sz);
  if (st != GDN_OK) return st;
  gdn::GateSrc gs;
  st = gate_source(io->g, io->beta, io->raw_gates, &gs);
  if (st != GDN_OK) return st;
  if (!io->qkv_pre || !io->z || !io->conv_w || !io->norm_w || !io->o || !io->S_T || !io->conv_T)
    return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {io->qkv_pre, io->z,      gs.g,      gs.beta, gs.a,     gs.b,
                        gs.A_log,    gs.dt_bias, io->conv_w, io->norm_w, io->S0, io->conv0,
                        io->o,       io->S_T,    io->conv_T, io->cu_seqlens, io->S_snap};
  if (!all_aligned(ptrs, 17)) return GDN_ERR_ALIGNMENT;
  Range in[12];
  int n = 0;
  in[n++] = range_of(io->qkv_pre, sz.qkv);
  in[n++] = range_of(io->z, sz.zo);
  n += gate_ranges(gs, sz, in + n);
  in[n++] = range_of(io->conv_w, sz.conv_w);
  in[n++] = range_of(io->norm_w, sz.norm_w);
  in[n++] = range_of(io->conv0, sz.conv);
  in[n++] = range_of(io->cu_seqlens, ((size_t)shape->B + 1) * sizeof(int));
  const int i_S0 = n;
  in[n++] = range_of(io->S0, sz.S);
  const Range ro = range_of(io->o, sz.zo), rs = range_of(io->S_T, sz.S), rc = range_of(io->conv_T, sz.conv),
              rp = range_of(io->S_snap, sz.snap);
  const bool in_place = io->S0 != nullptr && io->S0 == io->S_T;
  for (int i = 0; i < n; ++i) {
    if (overlap(ro, in[i]) || overlap(rc, in[i]) || overlap(rp, in[i])) return GDN_ERR_ALIAS;
    if (i == i_S0 && in_place) continue;
    if (overlap(rs, in[i])) return GDN_ERR_ALIAS;
  }
  if (overlap(ro, rs) || overlap(ro, rc) || overlap(rs, rc) || overlap(rp, ro) || overlap(rp, rs) ||
      overlap(rp, rc))
    return GDN_ERR_ALIAS;
  // bf16 io without snapshots: the chunked tensor-core kernel, with q^ and k^
  // staged through the workspace when one is given.  fp32 io (fp32
  // arithmetic throughout) and per-token snapshots: the token-serial kernel.
  const bool bf16 = shape->io_dtype == GDN_BF16;
  const bool chunked = bf16 && !io->S_snap;
  // With a workspace the chunked path takes the fastest form that fits it:
  // the chunk-parallel / sequential split (split_workspace_bytes), else the
  // staged q^ / k^ form (qk_workspace_bytes).
  void *ws = nullptr;
  bool split = false;
  gdn::SplitArgs sa{};
  if (chunked && io->workspace) {
    const size_t need_qk = qk_workspace_bytes(d, tokens);
    const size_t need_split = split_workspace_bytes(d, tokens, packed, &sa);
    if ((reinterpret_cast<uintptr_t>(io->workspace) & 255u) != 0) return GDN_ERR_ALIGNMENT;
    if (io->workspace_bytes < need_qk) return GDN_ERR_INVALID_ARG;
    split = need_split > 0 && io->workspace_bytes >= need_split && split_pays(d.B * d.Hv);
    const Range rw = range_of(io->workspace, split ? need_split : need_qk);
    for (int i = 0; i < n; ++i)
      if (overlap(rw, in[i])) return GDN_ERR_ALIAS;
    if (overlap(rw, ro) || overlap(rw, rs) || overlap(rw, rc)) return GDN_ERR_ALIAS;
    ws = io->workspace;
    if (split) {
      const long long items = (long long)sa.nslots * d.Hv;
      uint8_t *base = static_cast<uint8_t *>(ws) + align256(need_qk);
      sa.cu = io->cu_seqlens;
      sa.ws_u = reinterpret_cast<float *>(base);
      sa.ws_nw = base + (size_t)items * 32768;
      sa.ws_m = base + (size_t)items * (32768 + 16384);
      sa.ws_vec = reinterpret_cast<float *>(base + (size_t)items * (32768 + 16384 + 8192));
      sa.flags = reinterpret_cast<int *>(base + (size_t)items * (32768 + 16384 + 8192 + 512));
    }
  }
  unsigned int *err = nullptr;
  st = check_device(&err);
  if (st != GDN_OK) return st;
  gdn::PrefillArgs a{d,         io->qkv_pre, io->z,   gs,         io->conv_w,     io->norm_w, io->S0,
                     io->conv0, io->o,       io->S_T, io->conv_T, io->cu_seqlens, io->S_snap, ws,  err};
  cudaError_t e;
  if (!chunked) {
    e = gdn::launch_prefill(a, bf16, (cudaStream_t)stream);
  } else {
    e = ws ? gdn::launch_prefill_qk(a, (cudaStream_t)stream, sa.flags, split ? (long long)sa.nslots * d.Hv : 0)
           : cudaSuccess;
    if (e == cudaSuccess)
      e = split ? gdn::launch_prefill_split(a, sa, (cudaStream_t)stream)
                : gdn::launch_prefill_chunked(a, true, (cudaStream_t)stream);
  }
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status decode_impl(const gdn_shape *shape, const gdn_decode_io *io, void *stream) {
  if (!shape || !io) return GDN_ERR_INVALID_ARG;
  if (shape->B < 1 || shape->T < 1) return GDN_ERR_INVALID_ARG;
  const long long tokens = (long long)shape->B * shape->T;
  gdn::Dims d;
  Sizes sz;
  gdn_status st = check_shape(shape, tokens, &d, &sz);
  if (st != GDN_OK) return st;
  gdn::GateSrc gs;
  st = gate_source(io->g, io->beta, io->raw_gates, &gs);
  if (st != GDN_OK) return st;
  if (!io->qkv_pre || !io->z || !io->conv_w || !io->norm_w || !io->S || !io->conv_in || !io->conv_out ||
      !io->o)
    return GDN_ERR_INVALID_ARG;
  const void *ptrs[] = {io->qkv_pre, io->z,        gs.g,       gs.beta,    gs.a,  gs.b,
                        gs.A_log,    gs.dt_bias,   io->conv_w, io->norm_w, io->S, io->S_snap,
                        io->conv_in, io->conv_out, io->o};
  if (!all_aligned(ptrs, 15)) return GDN_ERR_ALIGNMENT;
  Range in[10];
  int n = 0;
  in[n++] = range_of(io->qkv_pre, sz.qkv);
  in[n++] = range_of(io->z, sz.zo);
  n += gate_ranges(gs, sz, in + n);
  in[n++] = range_of(io->conv_w, sz.conv_w);
  in[n++] = range_of(io->norm_w, sz.norm_w);
  in[n++] = range_of(io->conv_in, sz.conv);
  const Range rS = range_of(io->S, sz.S), ro = range_of(io->o, sz.zo), rc = range_of(io->conv_out, sz.conv),
              rp = range_of(io->S_snap, sz.snap);
  for (int i = 0; i < n; ++i)
    if (overlap(rS, in[i]) || overlap(ro, in[i]) || overlap(rc, in[i]) || overlap(rp, in[i]))
      return GDN_ERR_ALIAS;
  if (overlap(rS, ro) || overlap(rS, rc) || overlap(ro, rc) || overlap(rp, rS) || overlap(rp, ro) ||
      overlap(rp, rc))
    return GDN_ERR_ALIAS;
  unsigned int *err = nullptr;
  st = check_device(&err);
  if (st != GDN_OK) return st;

  const bool bf16 = shape->io_dtype == GDN_BF16;
  cudaError_t e;
  if (shape->T <= gdn::kDecodeMaxT) {
    gdn::DecodeArgs a{d,           io->qkv_pre,  io->z, gs, io->conv_w, io->norm_w, io->S, io->S_snap,
                      io->conv_in, io->conv_out, io->o, err};
    e = gdn::launch_decode(a, bf16, (cudaStream_t)stream);
  } else {
    // T tokens from the cache = a T-token prefill with the state in place.
    gdn::PrefillArgs a{d,     io->qkv_pre, io->z,        gs,      io->conv_w, io->norm_w, io->S, io->conv_in,
                       io->o, io->S,       io->conv_out, nullptr, io->S_snap, nullptr, err};
    e = gdn::launch_prefill(a, bf16, (cudaStream_t)stream);
  }
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
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
    case GDN_ERR_BOUNDS: return "device bounds check failed";
    default: return "unknown status";
  }
}

gdn_status gdn_prefill(const gdn_shape *shape, const void *qkv_pre, const void *z,
                       const float *g, const float *beta, const void *conv_w,
                       const void *norm_w, const float *S0, const void *conv0, void *o,
                       float *S_T, void *conv_T, void *stream) {
  if (!g || !beta) return GDN_ERR_INVALID_ARG;
  const gdn_prefill_io io{qkv_pre, z,  g,    beta,   nullptr, conv_w,  norm_w,
                          S0,      conv0, o, S_T, conv_T, nullptr, nullptr};
  return prefill_impl(shape, &io, stream);
}

gdn_status gdn_prefill_ex(const gdn_shape *shape, const gdn_prefill_io *io, void *stream) {
  return prefill_impl(shape, io, stream);
}

gdn_status gdn_prefill_static(const gdn_shape *shape, const gdn_prefill_io *io, void *stream) {
  if (!shape || !io || io->workspace) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_prefill_staged_bytes(shape, io->cu_seqlens != nullptr ? 1 : 0);
  if (need > GDN_STATIC_SCRATCH_BYTES) return GDN_ERR_UNSUPPORTED_SHAPE;
  // The device is checked before the scratch is looked up (which loads the
  // module), so that a wrong device reports GDN_ERR_NO_DEVICE as elsewhere.
  unsigned int *err = nullptr;
  const gdn_status dev_st = check_device(&err);
  if (dev_st != GDN_OK) return dev_st;
  gdn_prefill_io staged = *io;
  if (need > 0 && shape->io_dtype == GDN_BF16 && !io->S_snap) {  // the chunked kernel: stage q^ / k^
    void *p = nullptr;
    if (gdn::static_scratch(&p) != cudaSuccess) return GDN_ERR_CUDA;
    staged.workspace = p;
    staged.workspace_bytes = GDN_STATIC_SCRATCH_BYTES;
  }
  return prefill_impl(shape, &staged, stream);
}

size_t gdn_prefill_workspace_bytes(const gdn_shape *shape, int packed) {
  if (!shape || shape->B < 1 || shape->T < 1 || shape->io_dtype != GDN_BF16) return 0;
  const long long tokens = packed ? (long long)shape->T : (long long)shape->B * shape->T;
  gdn::Dims d;
  Sizes sz;
  if (check_shape(shape, tokens, &d, &sz) != GDN_OK) return 0;
  const size_t split = split_workspace_bytes(d, tokens, packed != 0);
  return split ? split : qk_workspace_bytes(d, tokens);
}

size_t gdn_prefill_staged_bytes(const gdn_shape *shape, int packed) {
  if (!shape || shape->B < 1 || shape->T < 1 || shape->io_dtype != GDN_BF16) return 0;
  const long long tokens = packed ? (long long)shape->T : (long long)shape->B * shape->T;
  gdn::Dims d;
  Sizes sz;
  if (check_shape(shape, tokens, &d, &sz) != GDN_OK) return 0;
  return qk_workspace_bytes(d, tokens);
}

gdn_status gdn_decode_step(const gdn_shape *shape, const void *qkv_pre, const void *z,
                           const float *g, const float *beta, const void *conv_w,
                           const void *norm_w, float *S, const void *conv_in, void *conv_out,
                           void *o, void *stream) {
  if (!shape || shape->T != 1 || !g || !beta) return GDN_ERR_INVALID_ARG;
  const gdn_decode_io io{qkv_pre, z, g, beta, nullptr, conv_w, norm_w, S, nullptr, conv_in, conv_out, o};
  return decode_impl(shape, &io, stream);
}

gdn_status gdn_decode_ex(const gdn_shape *shape, const gdn_decode_io *io, void *stream) {
  return decode_impl(shape, io, stream);
}

gdn_status gdn_linear(int M, int N, int K, const void *x, long long ldx, const void *w, long long ldw,
                      int n_out, const gdn_linear_out *out, void *stream) {
  if (M < 1 || N < 1 || K < 1 || !x || !w || !out || n_out < 1 || n_out > gdn::kGemmMaxOut)
    return GDN_ERR_INVALID_ARG;
  if (ldx < K || ldw < K) return GDN_ERR_INVALID_ARG;
  if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30) || ldx > (1LL << 32) || ldw > (1LL << 32))
    return GDN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w) || (ldx % 8) != 0 || (ldw % 8) != 0) return GDN_ERR_ALIGNMENT;
  gdn::GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.x = x;
  a.w = w;
  a.ldx = ldx;
  a.ldw = ldw;
  a.n_out = n_out;
  const Range rx = range_of(x, (size_t)(M - 1) * ldx * 2 + (size_t)K * 2);
  const Range rw = range_of(w, (size_t)(N - 1) * ldw * 2 + (size_t)K * 2);
  Range ro[gdn::kGemmMaxOut];
  for (int o = 0; o < n_out; ++o) {
    const gdn_linear_out &q = out[o];
    if (!q.ptr || q.col_begin < 0 || q.col_end <= q.col_begin || q.col_end > N || q.ld < q.col_end - q.col_begin)
      return GDN_ERR_INVALID_ARG;
    for (int p = 0; p < o; ++p)
      if (q.col_begin < out[p].col_end && out[p].col_begin < q.col_end) return GDN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q.ptr) & 1u) != 0) return GDN_ERR_ALIGNMENT;
    ro[o] = range_of(q.ptr, ((size_t)(M - 1) * q.ld + (size_t)(q.col_end - q.col_begin)) * 2);
    if (overlap(ro[o], rx) || overlap(ro[o], rw)) return GDN_ERR_ALIAS;
    for (int p = 0; p < o; ++p)
      if (overlap(ro[o], ro[p])) return GDN_ERR_ALIAS;
    a.out[o] = gdn::GemmOut{q.col_begin, q.col_end, q.ptr, q.ld,
                            aligned16(q.ptr) && (q.ld % 8) == 0 && (q.col_begin % 8) == 0 ? 1 : 0};
  }
  unsigned int *err = nullptr;
  gdn_status st = check_device(&err);
  if (st != GDN_OK) return st;
  a.err = err;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return GDN_ERR_CUDA;
  cudaError_t e = gdn::launch_gemm(a, sms, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_selftest_wait_timeout(int wait_us, void *stream) {
  if (wait_us < 1 || wait_us > 1000000) return GDN_ERR_INVALID_ARG;
  unsigned int *err = nullptr;
  gdn_status st = check_device(&err);
  if (st != GDN_OK) return st;
  cudaError_t e = gdn::launch_wait_selftest(err, 1000ull * (unsigned long long)wait_us, (cudaStream_t)stream);
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
  if (word & gdn::kErrTimeout) return GDN_ERR_TIMEOUT;
  if (word & gdn::kErrBounds) return GDN_ERR_BOUNDS;
  if (word & gdn::kErrSeqlens) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

}  // extern "C"
