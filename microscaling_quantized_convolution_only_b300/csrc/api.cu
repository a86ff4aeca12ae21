// api.cu -- the C ABI declared in include/mqconv.h: argument checks, launch
// planning and launches.  The library never allocates device memory.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>

#include "../../include/mqconv.h"
#include "kernels.h"

namespace {

// Device status word: kernels OR error bits into it; mqconv_device_status()
// reads and clears it.  One copy per device that loads the library.
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;
struct DevInfo {
  bool ready = false;
  uint32_t *status = nullptr;
  int num_sms = 0;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

mq_status dev_info(DevInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo &d = g_dev[dev];
  if (!d.ready) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MQ_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MQ_ERR_CUDA;
    d.status = static_cast<uint32_t *>(p);
    d.num_sms = sms;
    d.ready = true;
  }
  *out = &d;
  return MQ_OK;
}

// Fault injection of the failure-detection tests (mqconv_test_fault_inject).
std::atomic<int> g_inject{0};

bool fmt_ok(int32_t f) { return f == MQ_FMT_E2M1 || f == MQ_FMT_E2M3 || f == MQ_FMT_E4M3; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t out_dim(int64_t in, int64_t k, int64_t s, int64_t pad) { return (in + 2 * pad - k) / s + 1; }

mq_status check_packed(const mq_packed *t, int32_t role, int64_t d0, int64_t d1, int64_t d2, int64_t d3) {
  if (!t || !t->codes || !t->scales || !t->s_t) return MQ_ERR_INVALID_ARG;
  if (!fmt_ok(t->fmt) || t->role != role) return MQ_ERR_INVALID_ARG;
  if (t->dims[0] != d0 || t->dims[1] != d1 || t->dims[2] != d2 || t->dims[3] != d3) return MQ_ERR_INVALID_ARG;
  if (!aligned16(t->codes) || !aligned16(t->scales) || (reinterpret_cast<uintptr_t>(t->s_t) & 3u))
    return MQ_ERR_ALIGNMENT;
  if (t->decoded && t->role != MQ_ROLE_WEIGHT) return MQ_ERR_INVALID_ARG;
  if (!aligned16(t->decoded)) return MQ_ERR_ALIGNMENT;
  return MQ_OK;
}

mq_status check_desc(const mq_conv_desc *d) {
  if (!d) return MQ_ERR_INVALID_ARG;
  if (d->N <= 0 || d->Cin <= 0 || d->Cout <= 0 || d->H <= 0 || d->W <= 0 || d->Kh <= 0 || d->Kw <= 0 ||
      d->stride <= 0 || d->pad < 0)
    return MQ_ERR_INVALID_ARG;
  if (d->N % 8 || d->Cin % 8 || d->Cout % 8) return MQ_ERR_UNSUPPORTED;
  const int64_t Ho = out_dim(d->H, d->Kh, d->stride, d->pad), Wo = out_dim(d->W, d->Kw, d->stride, d->pad);
  if (Ho <= 0 || Wo <= 0) return MQ_ERR_INVALID_ARG;
  // the kernels index positions, block groups and columns with 32-bit integers
  const int64_t lim = INT_MAX / 16;
  if (d->H * d->W * (d->N / 8) > lim || Ho * Wo * (d->N / 8) > lim || d->Kh * d->Kw * d->Cin > lim ||
      d->Cin > 65536 || d->Cout > 65536 || d->stride > 16 || d->Kh > 64 || d->Kw > 64)
    return MQ_ERR_UNSUPPORTED;
  return MQ_OK;
}

mq::ConvParams base_params(const mq_conv_desc *d, int op, uint32_t *status) {
  mq::ConvParams p;
  std::memset(&p, 0, sizeof(p));
  p.op = op;
  p.N = (int)d->N;
  p.Cin = (int)d->Cin;
  p.H = (int)d->H;
  p.W = (int)d->W;
  p.Cout = (int)d->Cout;
  p.Kh = (int)d->Kh;
  p.Kw = (int)d->Kw;
  p.stride = (int)d->stride;
  p.pad = (int)d->pad;
  p.Ho = (int)out_dim(d->H, d->Kh, d->stride, d->pad);
  p.Wo = (int)out_dim(d->W, d->Kw, d->stride, d->pad);
  p.NG = p.N / 8;
  p.CIG = p.Cin / 8;
  p.COG = p.Cout / 8;
  p.status = status;
  p.inject = g_inject.load();
  return p;
}

mq::Operand operand(const mq_packed *t) {
  mq::Operand o;
  o.codes = static_cast<const uint8_t *>(t->codes);
  o.scales = t->scales;
  o.s_t = t->s_t;
  o.fmt = t->fmt;
  return o;
}

float pre_mult(int fa, int fb) { return (fa == MQ_FMT_E4M3 ? 4.0f : 1.0f) * (fb == MQ_FMT_E4M3 ? 4.0f : 1.0f); }

// Forward or data gradient: the halo-reuse kernel when the layer fits it
// (stride 1), the generic implicit-im2col kernel otherwise.
mq_status run_conv(mq::ConvParams &p, int num_sms, cudaStream_t s) {
  mq::HaloConv h;
  if (mq::halo_plan(p, h, num_sms)) return mq::halo_launch(p, h, num_sms, s) == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
  mq::conv_plan(p);
  return mq::launch_conv(p, num_sms, s) == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

// Split-K partial sums of one plan.
size_t partial_bytes(int splits, const mq::ConvParams &p) {
  return (size_t)splits * (size_t)p.Cout * (size_t)(p.Kh * p.Kw * p.Cin) * sizeof(float);
}

// Workspace of the weight gradient: enough for every plan the call may pick
// whatever the element formats (the halo kernel's tiling depends on them).
size_t wgrad_ws_bytes(const mq_conv_desc *d) {
  mq::ConvParams p = base_params(d, mq::OP_WGRAD, nullptr);
  mq::conv_plan(p);
  size_t need = partial_bytes(p.k_splits, p);
  for (int f : {MQ_FMT_E2M1, MQ_FMT_E2M3, MQ_FMT_E4M3}) {
    mq::ConvParams q = base_params(d, mq::OP_WGRAD, nullptr);
    q.a.fmt = q.b.fmt = f;
    mq::HaloWgrad h;
    if (mq::halo_wgrad_plan(q, h, 0)) need = std::max(need, partial_bytes(h.splits, q));
  }
  return need;
}

// Weight gradient into the split-K buffer `partials`, then the fixed-order
// reduction into dW.  max_splits bounds the split count (0: none).
mq_status run_wgrad(mq::ConvParams &p, float *partials, size_t bytes, int max_splits, float *dw, int num_sms,
                    cudaStream_t s) {
  p.out = partials;
  mq::HaloWgrad h;
  if (mq::halo_wgrad_plan(p, h, max_splits)) {
    if (partial_bytes(h.splits, p) > bytes) return MQ_ERR_WORKSPACE;
    if (mq::halo_wgrad_launch(p, h, num_sms, s) != cudaSuccess) return MQ_ERR_CUDA;
    p.k_splits = h.splits;
    p.ncols = h.ncols;
  } else {
    mq::conv_plan(p);
    if (max_splits > 0 && p.k_splits > max_splits) {
      int per = (p.kg_total + max_splits - 1) / max_splits;
      per = (per + mq::CONV_KCH - 1) / mq::CONV_KCH * mq::CONV_KCH;
      p.kg_per_split = per;
      p.k_splits = (p.kg_total + per - 1) / per;
    }
    if (partial_bytes(p.k_splits, p) > bytes) return MQ_ERR_WORKSPACE;
    if (mq::launch_conv(p, num_sms, s) != cudaSuccess) return MQ_ERR_CUDA;
  }
  if (mq::launch_wgrad_reduce(p, dw, s) != cudaSuccess) return MQ_ERR_CUDA;
  return MQ_OK;
}

}  // namespace

// ------------------------------------------------ wgrad without allocation
// Fixed device scratch for mqconv_wgrad_noalloc: it holds the split-K partial
// sums that mqconv_wgrad keeps in a caller-supplied workspace.  Every device
// that loads this library reserves it until the process exits.  Host code must
// not pass the symbol itself to a kernel (on the host it names a stand-in, not
// device memory); its device address is looked up per device below.
static __device__ __align__(256) float g_wgrad_scratch[MQCONV_WGRAD_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

float *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_wgrad_scratch on the current device, looked up on the
// first call per device (with that device current).
mq_status scratch_addr(float **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_wgrad_scratch) != cudaSuccess || !ptr) return MQ_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<float *>(ptr);
  }
  *out = g_scratch_addr[dev];
  return MQ_OK;
}

// Forward (a = Xq) or data gradient (a = dYq) with optional fused
// requantization of the fp32 result into packed blocks.
mq_status conv_fwd_or_dgrad(int op, const mq_conv_desc *desc, const mq_packed *a, const mq_packed *wq, float *out,
                            const mq_requant *rq, mq_stream stream) {
  mq_status st = check_desc(desc);
  if (st != MQ_OK) return st;
  const int64_t Ho = out_dim(desc->H, desc->Kh, desc->stride, desc->pad);
  const int64_t Wo = out_dim(desc->W, desc->Kw, desc->stride, desc->pad);
  const bool fwd = op == mq::OP_FWD;
  if (fwd) {
    if ((st = check_packed(a, MQ_ROLE_ACT, desc->N, desc->Cin, desc->H, desc->W)) != MQ_OK) return st;
  } else {
    if ((st = check_packed(a, MQ_ROLE_GRAD, desc->N, desc->Cout, Ho, Wo)) != MQ_OK) return st;
  }
  if ((st = check_packed(wq, MQ_ROLE_WEIGHT, desc->Cout, desc->Cin, desc->Kh, desc->Kw)) != MQ_OK) return st;
  if (!out && !rq) return MQ_ERR_INVALID_ARG;
  if (out && !aligned16(out)) return MQ_ERR_ALIGNMENT;
  if (rq) {
    if (!rq->amax_in || !fmt_ok(rq->fmt) || !rq->out || rq->out->fmt != rq->fmt) return MQ_ERR_INVALID_ARG;
    if (rq->rounding != MQ_ROUND_RN && rq->rounding != MQ_ROUND_SR) return MQ_ERR_INVALID_ARG;
    st = fwd ? check_packed(rq->out, MQ_ROLE_ACT, desc->N, desc->Cout, Ho, Wo)
             : check_packed(rq->out, MQ_ROLE_GRAD, desc->N, desc->Cin, desc->H, desc->W);
    if (st != MQ_OK) return st;
    if ((reinterpret_cast<uintptr_t>(rq->amax_in) & 3u) ||
        (rq->amax_out && (reinterpret_cast<uintptr_t>(rq->amax_out) & 3u)))
      return MQ_ERR_ALIGNMENT;
  }
  DevInfo *di = nullptr;
  if ((st = dev_info(&di)) != MQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mq::ConvParams p = base_params(desc, op, di->status);
  p.a = operand(a);
  p.b = operand(wq);
  p.pre_mult = pre_mult(a->fmt, wq->fmt);
  p.out = out;
  p.wdec = wq->decoded;
  if (rq) {
    p.rq.codes = static_cast<uint8_t *>(rq->out->codes);
    p.rq.scales = rq->out->scales;
    p.rq.s_t_out = rq->out->s_t;
    p.rq.amax_in = rq->amax_in;
    p.rq.amax_out_bits = reinterpret_cast<uint32_t *>(rq->amax_out);
    p.rq.fmt = rq->fmt;
    p.rq.sr = rq->rounding == MQ_ROUND_SR ? 1 : 0;
    p.rq.sr_seed = rq->sr_seed;
    if (rq->amax_out && cudaMemsetAsync(rq->amax_out, 0, sizeof(float), s) != cudaSuccess) return MQ_ERR_CUDA;
  }
  return run_conv(p, di->num_sms, s);
}

}  // namespace

extern "C" {

int32_t mqconv_abi_version(void) { return MQCONV_ABI_VERSION; }

const char *mqconv_status_string(mq_status s) {
  switch (s) {
    case MQ_OK: return "ok";
    case MQ_ERR_INVALID_ARG: return "invalid argument";
    case MQ_ERR_UNSUPPORTED: return "unsupported shape (batch and channels must be multiples of 8)";
    case MQ_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case MQ_ERR_NONFINITE: return "non-finite value in a quantized input";
    case MQ_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
    case MQ_ERR_CUDA: return "CUDA runtime error";
    case MQ_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

size_t mqconv_packed_code_bytes(int32_t fmt, const int64_t dims[4]) {
  if (!dims || !fmt_ok(fmt) || dims[0] <= 0 || dims[1] <= 0 || dims[2] <= 0 || dims[3] <= 0 || dims[0] % 8 ||
      dims[1] % 8)
    return 0;
  return (size_t)(dims[0] / 8) * (size_t)(dims[1] / 8) * (size_t)dims[2] * (size_t)dims[3] *
         (size_t)mq::block_bytes(fmt);
}

size_t mqconv_weight_decoded_bytes(const int64_t dims[4]) { return 128 * mqconv_packed_scale_bytes(dims); }

mq_status mqconv_weight_decode(const mq_packed *wq, mq_stream stream) {
  if (!wq || !wq->decoded || wq->role != MQ_ROLE_WEIGHT) return MQ_ERR_INVALID_ARG;
  const int64_t *d = wq->dims;
  if (d[0] <= 0 || d[1] <= 0 || d[2] <= 0 || d[3] <= 0) return MQ_ERR_INVALID_ARG;
  if (d[0] % 8 || d[1] % 8) return MQ_ERR_UNSUPPORTED;
  mq_status st = check_packed(wq, MQ_ROLE_WEIGHT, d[0], d[1], d[2], d[3]);
  if (st != MQ_OK) return st;
  DevInfo *di = nullptr;
  if ((st = dev_info(&di)) != MQ_OK) return st;
  return mq::launch_weight_decode(static_cast<const uint8_t *>(wq->codes), wq->scales, wq->fmt,
                                  (d[0] / 8) * (d[1] / 8) * d[2] * d[3], wq->decoded, di->num_sms,
                                  reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MQ_OK
             : MQ_ERR_CUDA;
}

size_t mqconv_packed_scale_bytes(const int64_t dims[4]) {
  if (!dims || dims[0] <= 0 || dims[1] <= 0 || dims[2] <= 0 || dims[3] <= 0 || dims[0] % 8 || dims[1] % 8) return 0;
  return (size_t)(dims[0] / 8) * (size_t)(dims[1] / 8) * (size_t)dims[2] * (size_t)dims[3];
}

namespace {
mq_status quantize_cbf(const void *src, int32_t dtype, int32_t layout, const mq_packed *dst, const float *amax_in,
                       float *amax_out, int sr, uint64_t seed, mq_stream stream) {
  if (!src || !dst || !dst->codes || !dst->scales || !dst->s_t) return MQ_ERR_INVALID_ARG;
  if (!fmt_ok(dst->fmt) || (dtype != MQ_DT_F32 && dtype != MQ_DT_BF16)) return MQ_ERR_INVALID_ARG;
  if (dst->role != MQ_ROLE_ACT && dst->role != MQ_ROLE_WEIGHT && dst->role != MQ_ROLE_GRAD) return MQ_ERR_INVALID_ARG;
  if (layout != MQ_LAYOUT_NCHW && layout != MQ_LAYOUT_HWCN && layout != MQ_LAYOUT_OIHW) return MQ_ERR_INVALID_ARG;
  if ((dst->role == MQ_ROLE_WEIGHT) != (layout == MQ_LAYOUT_OIHW)) return MQ_ERR_INVALID_ARG;
  if (dst->decoded && dst->role != MQ_ROLE_WEIGHT) return MQ_ERR_INVALID_ARG;
  const int64_t *d = dst->dims;
  if (d[0] <= 0 || d[1] <= 0 || d[2] <= 0 || d[3] <= 0) return MQ_ERR_INVALID_ARG;
  if (d[0] % 8 || d[1] % 8) return MQ_ERR_UNSUPPORTED;
  if (!amax_in && !amax_out) return MQ_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst->codes) || !aligned16(dst->decoded) ||
      (reinterpret_cast<uintptr_t>(dst->s_t) & 3u) ||
      (amax_in && (reinterpret_cast<uintptr_t>(amax_in) & 3u)) ||
      (amax_out && (reinterpret_cast<uintptr_t>(amax_out) & 3u)))
    return MQ_ERR_ALIGNMENT;
  const int64_t n = d[0] * d[1] * d[2] * d[3];
  if (n / d[0] / d[1] != d[2] * d[3] || n > (int64_t)1 << 40) return MQ_ERR_UNSUPPORTED;

  DevInfo *di = nullptr;
  mq_status st = dev_info(&di);
  if (st != MQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  mq::QuantParams p;
  p.d0 = d[0];
  p.d1 = d[1];
  p.d2 = d[2];
  p.d3 = d[3];
  p.codes = static_cast<uint8_t *>(dst->codes);
  p.scales = dst->scales;
  p.s_t_out = dst->s_t;
  p.status = di->status;
  p.sr = sr;
  p.sr_seed = seed;
  if (!amax_in) {
    uint32_t *bits = reinterpret_cast<uint32_t *>(amax_out);
    if (cudaMemsetAsync(bits, 0, sizeof(uint32_t), s) != cudaSuccess) return MQ_ERR_CUDA;
    if (mq::launch_amax(src, dtype, n, bits, di->num_sms, s) != cudaSuccess) return MQ_ERR_CUDA;
    p.amax_src_bits = bits;
    p.amax_meas_bits = nullptr;
  } else {
    p.amax_src_bits = reinterpret_cast<const uint32_t *>(amax_in);
    p.amax_meas_bits = reinterpret_cast<uint32_t *>(amax_out);
    if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess) return MQ_ERR_CUDA;
  }
  if (mq::launch_quantize(src, dtype, layout, dst->fmt, p, di->num_sms, s) != cudaSuccess) return MQ_ERR_CUDA;
  if (dst->decoded &&
      mq::launch_weight_decode(p.codes, p.scales, dst->fmt, (d[0] / 8) * (d[1] / 8) * d[2] * d[3], dst->decoded,
                               di->num_sms, s) != cudaSuccess)
    return MQ_ERR_CUDA;
  return MQ_OK;
}
}  // namespace

mq_status mqconv_quantize_cbf(const void *src, int32_t dtype, int32_t layout, const mq_packed *dst,
                              const float *amax_in, float *amax_out, mq_stream stream) {
  return quantize_cbf(src, dtype, layout, dst, amax_in, amax_out, 0, 0, stream);
}

mq_status mqconv_quantize_cbf_sr(const void *src, int32_t dtype, int32_t layout, const mq_packed *dst,
                                 const float *amax_in, float *amax_out, uint64_t seed, mq_stream stream) {
  return quantize_cbf(src, dtype, layout, dst, amax_in, amax_out, 1, seed, stream);
}

mq_status mqconv_fwd(const mq_conv_desc *desc, const mq_packed *xq, const mq_packed *wq, float *y,
                     const mq_requant *rq, mq_stream stream) {
  return conv_fwd_or_dgrad(mq::OP_FWD, desc, xq, wq, y, rq, stream);
}

mq_status mqconv_dgrad(const mq_conv_desc *desc, const mq_packed *wq, const mq_packed *dyq, float *dx,
                       mq_stream stream) {
  if (!dx) return MQ_ERR_INVALID_ARG;
  return conv_fwd_or_dgrad(mq::OP_DGRAD, desc, dyq, wq, dx, nullptr, stream);
}

mq_status mqconv_dgrad_requant(const mq_conv_desc *desc, const mq_packed *wq, const mq_packed *dyq, float *dx,
                               const mq_requant *rq, mq_stream stream) {
  if (!rq) return MQ_ERR_INVALID_ARG;
  return conv_fwd_or_dgrad(mq::OP_DGRAD, desc, dyq, wq, dx, rq, stream);
}

size_t mqconv_wgrad_workspace_bytes(const mq_conv_desc *desc) {
  if (check_desc(desc) != MQ_OK) return 0;
  return wgrad_ws_bytes(desc);
}

mq_status mqconv_wgrad(const mq_conv_desc *desc, const mq_packed *dyq, const mq_packed *xq, float *dw,
                       void *workspace, size_t ws_bytes, mq_stream stream) {
  mq_status st = check_desc(desc);
  if (st != MQ_OK) return st;
  const int64_t Ho = out_dim(desc->H, desc->Kh, desc->stride, desc->pad);
  const int64_t Wo = out_dim(desc->W, desc->Kw, desc->stride, desc->pad);
  if ((st = check_packed(dyq, MQ_ROLE_GRAD, desc->N, desc->Cout, Ho, Wo)) != MQ_OK) return st;
  if ((st = check_packed(xq, MQ_ROLE_ACT, desc->N, desc->Cin, desc->H, desc->W)) != MQ_OK) return st;
  if (!dw) return MQ_ERR_INVALID_ARG;
  if (!aligned16(dw)) return MQ_ERR_ALIGNMENT;
  if (!workspace || ws_bytes < wgrad_ws_bytes(desc)) return MQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MQ_ERR_ALIGNMENT;
  DevInfo *di = nullptr;
  if ((st = dev_info(&di)) != MQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mq::ConvParams p = base_params(desc, mq::OP_WGRAD, di->status);
  p.a = operand(dyq);
  p.b = operand(xq);
  p.pre_mult = pre_mult(dyq->fmt, xq->fmt);
  return run_wgrad(p, static_cast<float *>(workspace), ws_bytes, 0, dw, di->num_sms, s);
}

mq_status mqconv_wgrad_noalloc(const mq_conv_desc *desc, const mq_packed *dyq, const mq_packed *xq, float *dw,
                               mq_stream stream) {
  mq_status st = check_desc(desc);
  if (st != MQ_OK) return st;
  const int64_t Ho = out_dim(desc->H, desc->Kh, desc->stride, desc->pad);
  const int64_t Wo = out_dim(desc->W, desc->Kw, desc->stride, desc->pad);
  if ((st = check_packed(dyq, MQ_ROLE_GRAD, desc->N, desc->Cout, Ho, Wo)) != MQ_OK) return st;
  if ((st = check_packed(xq, MQ_ROLE_ACT, desc->N, desc->Cin, desc->H, desc->W)) != MQ_OK) return st;
  if (!dw) return MQ_ERR_INVALID_ARG;
  if (!aligned16(dw)) return MQ_ERR_ALIGNMENT;
  DevInfo *di = nullptr;
  if ((st = dev_info(&di)) != MQ_OK) return st;
  mq::ConvParams p = base_params(desc, mq::OP_WGRAD, di->status);
  p.a = operand(dyq);
  p.b = operand(xq);
  p.pre_mult = pre_mult(dyq->fmt, xq->fmt);
  // fit the split-K partial sums into the fixed scratch: fewer, longer splits
  const size_t per_split = partial_bytes(1, p);
  const size_t max_splits = MQCONV_WGRAD_NOALLOC_SCRATCH_BYTES / per_split;
  if (max_splits == 0) return MQ_ERR_WORKSPACE;
  float *scratch = nullptr;
  if ((st = scratch_addr(&scratch)) != MQ_OK) return st;
  return run_wgrad(p, scratch, MQCONV_WGRAD_NOALLOC_SCRATCH_BYTES, (int)std::min<size_t>(max_splits, 1 << 20), dw,
                   di->num_sms, reinterpret_cast<cudaStream_t>(stream));
}

mq_status mqconv_test_fault_inject(int32_t what) {
  if (what != MQ_INJECT_NONE && what != MQ_INJECT_WITHHOLD_ACC_RELEASE) return MQ_ERR_INVALID_ARG;
  static_assert(MQ_INJECT_WITHHOLD_ACC_RELEASE == mq::INJECT_WITHHOLD_ACC_RELEASE, "injection codes");
  g_inject.store(what);
  return MQ_OK;
}

mq_status mqconv_device_status(mq_stream stream, int32_t *host_status) {
  if (!host_status) return MQ_ERR_INVALID_ARG;
  DevInfo *di = nullptr;
  mq_status st = dev_info(&di);
  if (st != MQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, di->status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MQ_ERR_CUDA;
  if (cudaMemsetAsync(di->status, 0, sizeof(uint32_t), s) != cudaSuccess) return MQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MQ_ERR_CUDA;
  *host_status = (int32_t)v;
  return MQ_OK;
}

}  // extern "C"
