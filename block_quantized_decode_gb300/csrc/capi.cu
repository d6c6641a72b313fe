// capi.cu -- the extern "C" boundary of libmlq (declared in include/mlq.h).
//
// Every entry point validates its arguments on the host first (status codes
// as in the page "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 6
// "Error handling": return a status, never abort), then checks the device
// (compute capability 10.3, cached per device), then queues one kernel on
// the caller's stream.  Nothing here allocates device memory.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mlq.h"
#include "mlq_launch.h"

namespace {

// Device status word: kernels record MLQ_E_TIMEOUT here when a bounded wait
// gives up.  One instance per device (a __device__ variable lives in every
// context that loads the module); its address is looked up once per device.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;

struct DevInfo {
  std::atomic<int> state{0};  // 0 = unknown, 1 = usable, 2 = unusable
  int num_sms = 0;
  int *status = nullptr;
};

DevInfo g_dev[kMaxDevices];
std::mutex g_init_mu;
std::atomic<unsigned long long> g_wait_ns{1000000000ull};
std::atomic<int> g_pdl{-1};
std::atomic<int> g_early{-1};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool pdl_enabled() {
  int v = g_pdl.load(std::memory_order_relaxed);
  if (v < 0) {
    const char *e = std::getenv("MLQ_PDL");
    v = (e != nullptr && std::strcmp(e, "0") == 0) ? 0 : 1;
    g_pdl.store(v, std::memory_order_relaxed);
  }
  return v == 1;
}

bool early_enabled() {
  int v = g_early.load(std::memory_order_relaxed);
  if (v < 0) {
    const char *e = std::getenv("MLQ_STATIC_WEIGHTS");
    v = (e != nullptr && std::strcmp(e, "1") == 0) ? 1 : 0;
    g_early.store(v, std::memory_order_relaxed);
  }
  return v == 1;
}

// Compute capability of `dev`; MLQ_FAKE_CC="major.minor" overrides it (a
// host-side test hook for the architecture guard).
bool query_cc(int dev, int *major, int *minor) {
  const char *fake = std::getenv("MLQ_FAKE_CC");
  if (fake != nullptr) {
    char *end = nullptr;
    *major = static_cast<int>(std::strtol(fake, &end, 10));
    *minor = (end != nullptr && *end == '.') ? static_cast<int>(std::strtol(end + 1, nullptr, 10)) : 0;
    return true;
  }
  if (cudaDeviceGetAttribute(major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
  return true;
}

mlq_status device_info(DevInfo **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLQ_E_ARCH;
  }
  DevInfo &d = g_dev[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    std::lock_guard<std::mutex> lk(g_init_mu);
    st = d.state.load(std::memory_order_acquire);
    if (st == 0) {
      int major = 0, minor = 0, sms = 0;
      bool ok = query_cc(dev, &major, &minor) && major == 10 && minor == 3;
      ok = ok && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
      int *status = nullptr;
      ok = ok && cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_device_status) == cudaSuccess;
      if (!ok) cudaGetLastError();
      d.num_sms = sms;
      d.status = status;
      st = ok ? 1 : 2;
      d.state.store(st, std::memory_order_release);
    }
  }
  if (st != 1) return MLQ_E_ARCH;
  *out = &d;
  return MLQ_OK;
}

mlq_status make_ctx(mlq::LaunchCtx *ctx, void *stream) {
  DevInfo *d = nullptr;
  mlq_status s = device_info(&d);
  if (s != MLQ_OK) return s;
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->pdl = pdl_enabled();
  ctx->num_sms = d->num_sms;
  ctx->status = d->status;
  ctx->wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  ctx->early_weights = ctx->pdl && early_enabled();
  return MLQ_OK;
}

mlq_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MLQ_OK;
  cudaGetLastError();
  return MLQ_E_CUDA;
}

bool cols_ok(int cols) { return cols > 0 && cols % MLQ_QK == 0 && cols <= MLQ_MAX_COLS; }

// Checks common to every product with a weight tensor.
mlq_status check_weights(const mlq_qtensor *W, const mlq_qact *x, int r0, int r1) {
  if (W == nullptr || x == nullptr) return MLQ_E_NULL;
  if (W->q == nullptr || W->d == nullptr || x->q == nullptr || x->d == nullptr) return MLQ_E_NULL;
  if (W->type != MLQ_Q4_0 && W->type != MLQ_Q8_0) return MLQ_E_TYPE;
  if (!cols_ok(W->cols) || W->rows < 0 || x->n != W->cols) return MLQ_E_SHAPE;
  if (r0 < 0 || r1 < r0 || r1 > W->rows) return MLQ_E_SHAPE;
  if (!aligned(W->q, 16) || !aligned(W->d, 16) || !aligned(x->q, 16) || !aligned(x->d, 16))
    return MLQ_E_ALIGN;
  return MLQ_OK;
}

mlq_status matvec_common(float *y, int32_t *sumi, const mlq_qtensor *W, const mlq_qact *x,
                         int r0, int r1, void *stream, int want_type) {
  if (y == nullptr && sumi == nullptr) return MLQ_E_NULL;
  mlq_status s = check_weights(W, x, r0, r1);
  if (s != MLQ_OK) return s;
  if (want_type >= 0 && W->type != want_type) return MLQ_E_TYPE;
  if (x->m != 1) return MLQ_E_SHAPE;
  if (!aligned(y != nullptr ? static_cast<const void *>(y) : static_cast<const void *>(sumi), 4))
    return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_matvec_m1(ctx, W->type, W->q, W->d, W->cols / MLQ_QK, x->q, x->d,
                                         y, sumi, r0, r1));
}

// Host-side checks and marshalling of a chain (everything but the workspace).
mlq_status build_chain_args(const mlq_chain_phase *phases, int nphases,
                            const mlq_chain_product *products, int nproducts,
                            mlq::ChainArgs *a) {
  if (phases == nullptr || products == nullptr) return MLQ_E_NULL;
  if (nphases < 1 || nphases > MLQ_CHAIN_MAX_PHASES) return MLQ_E_SHAPE;
  if (nproducts < 1 || nproducts > MLQ_CHAIN_MAX_PRODUCTS) return MLQ_E_SHAPE;
  const uint8_t type = products[0].W.type;
  for (int j = 0; j < nproducts; ++j) {
    const mlq_chain_product &p = products[j];
    if (p.W.rows > 0 && (p.W.q == nullptr || p.W.d == nullptr || p.y == nullptr)) return MLQ_E_NULL;
    if (p.W.type != MLQ_Q4_0 && p.W.type != MLQ_Q8_0) return MLQ_E_TYPE;
    if (p.W.type != type) return MLQ_E_TYPE;
    if (!cols_ok(p.W.cols) || p.W.cols % 128 != 0 || p.W.rows < 0) return MLQ_E_SHAPE;
    if (!aligned(p.W.q, 16) || !aligned(p.W.d, 16) || !aligned(p.y, 4)) return MLQ_E_ALIGN;
    a->prod[j].wq = static_cast<const uint8_t *>(p.W.q);
    a->prod[j].wd = p.W.d;
    a->prod[j].y = p.y;
    a->prod[j].rows = p.W.rows;
  }
  int kmax = 0;
  for (int i = 0; i < nphases; ++i) {
    const mlq_chain_phase &ph = phases[i];
    if (ph.x == nullptr) return MLQ_E_NULL;
    if ((ph.xq_out == nullptr) != (ph.xd_out == nullptr)) return MLQ_E_NULL;
    if (ph.count < 1 || ph.first < 0 || ph.first > nproducts - ph.count) return MLQ_E_SHAPE;
    if (!cols_ok(ph.n) || ph.n % 128 != 0) return MLQ_E_SHAPE;
    for (int j = ph.first; j < ph.first + ph.count; ++j)
      if (products[j].W.cols != ph.n) return MLQ_E_SHAPE;
    if (!aligned(ph.x, 16) || !aligned(ph.xq_out, 16) || !aligned(ph.xd_out, 16))
      return MLQ_E_ALIGN;
    a->phase[i].x = ph.x;
    a->phase[i].xq_out = ph.xq_out;
    a->phase[i].xd_out = ph.xd_out;
    a->phase[i].nb = ph.n / MLQ_QK;
    a->phase[i].first = ph.first;
    a->phase[i].count = ph.count;
    if (ph.n > kmax) kmax = ph.n;
  }
  a->nphases = nphases;
  a->kmax = kmax;
  return MLQ_OK;
}

}  // namespace

namespace mlq {
void prefer_max_shared_impl(const void *kern) {
  static std::mutex mu;
  static const void *seen[256];
  static int nseen = 0;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < nseen; ++i)
    if (seen[i] == kern) return;
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                       cudaSharedmemCarveoutMaxShared);
  cudaGetLastError();
  if (nseen < 256) seen[nseen++] = kern;
}
}  // namespace mlq

extern "C" {

mlq_status mlq_init(void) {
  DevInfo *d = nullptr;
  return device_info(&d);
}

mlq_status mlq_quantize_q8(mlq_qact *out, const float *x, int k, void *stream) {
  mlq::diag_entry("mlq_quantize_q8", "k=%d m=%d", k, out ? out->m : -1);
  if (out == nullptr || x == nullptr || out->q == nullptr || out->d == nullptr) return MLQ_E_NULL;
  if (!cols_ok(k) || out->n != k || out->m < 1) return MLQ_E_SHAPE;
  if (!aligned(x, 16) || !aligned(out->q, 16) || !aligned(out->d, 16)) return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_quantize_q8(ctx, x, out->q, out->d, out->m, k));
}

mlq_status mlq_matvec_q4(float *y, const mlq_qtensor *W, const mlq_qact *x, int r0, int r1,
                         void *stream) {
  mlq::diag_entry("mlq_matvec_q4", "rows=%d cols=%d r=[%d,%d)", W ? W->rows : -1, W ? W->cols : -1, r0, r1);
  if (y == nullptr) return MLQ_E_NULL;
  return matvec_common(y, nullptr, W, x, r0, r1, stream, MLQ_Q4_0);
}

mlq_status mlq_matvec_q8(float *y, const mlq_qtensor *W, const mlq_qact *x, int r0, int r1,
                         void *stream) {
  mlq::diag_entry("mlq_matvec_q8", "rows=%d cols=%d r=[%d,%d)", W ? W->rows : -1, W ? W->cols : -1, r0, r1);
  if (y == nullptr) return MLQ_E_NULL;
  return matvec_common(y, nullptr, W, x, r0, r1, stream, MLQ_Q8_0);
}

mlq_status mlq_block_sumi(int32_t *sumi, const mlq_qtensor *W, const mlq_qact *x, int r0, int r1,
                          void *stream) {
  mlq::diag_entry("mlq_block_sumi", "rows=%d cols=%d r=[%d,%d)", W ? W->rows : -1, W ? W->cols : -1, r0, r1);
  if (sumi == nullptr) return MLQ_E_NULL;
  return matvec_common(nullptr, sumi, W, x, r0, r1, stream, -1);
}

mlq_status mlq_gemm_q4_small_m(float *Y, int ldy, const mlq_qtensor *W, const mlq_qact *X, int M,
                               int r0, int r1, void *stream) {
  mlq::diag_entry("mlq_gemm_q4_small_m", "M=%d rows=%d cols=%d r=[%d,%d)", M, W ? W->rows : -1, W ? W->cols : -1, r0, r1);
  if (Y == nullptr) return MLQ_E_NULL;
  mlq_status s = check_weights(W, X, r0, r1);
  if (s != MLQ_OK) return s;
  if (W->type != MLQ_Q4_0) return MLQ_E_TYPE;
  if (M < 1 || M > MLQ_MAX_M || X->m != M || ldy < r1 || ldy < 1) return MLQ_E_SHAPE;
  if (!aligned(Y, 4)) return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_gemm_q4_small_m(ctx, W->q, W->d, W->cols / MLQ_QK, X->q, X->d, M,
                                               Y, ldy, r0, r1, W->rows));
}

mlq_status mlq_matvec_fused(const float *x, int n, const mlq_chain_product *products,
                            int nproducts, int8_t *xq_out, float *xd_out, unsigned flags,
                            void *stream) {
  mlq::diag_entry("mlq_matvec_fused", "n=%d products=%d", n, nproducts);
  if (x == nullptr || products == nullptr) return MLQ_E_NULL;
  if ((xq_out == nullptr) != (xd_out == nullptr)) return MLQ_E_NULL;
  if (nproducts < 1 || nproducts > MLQ_FUSED_MAX_PRODUCTS || !cols_ok(n)) return MLQ_E_SHAPE;
  if (!aligned(x, 16) || !aligned(xq_out, 16) || !aligned(xd_out, 16)) return MLQ_E_ALIGN;
  mlq::FusedArgs a = {};
  const uint8_t type = products[0].W.type;
  for (int j = 0; j < nproducts; ++j) {
    const mlq_chain_product &p = products[j];
    if (p.W.rows > 0 && (p.W.q == nullptr || p.W.d == nullptr || p.y == nullptr)) return MLQ_E_NULL;
    if (p.W.type != MLQ_Q4_0 && p.W.type != MLQ_Q8_0) return MLQ_E_TYPE;
    if (p.W.type != type) return MLQ_E_TYPE;
    if (p.W.cols != n || p.W.rows < 0) return MLQ_E_SHAPE;
    if (!aligned(p.W.q, 16) || !aligned(p.W.d, 16) || !aligned(p.y, 4)) return MLQ_E_ALIGN;
    a.prod[j].wq = static_cast<const uint8_t *>(p.W.q);
    a.prod[j].wd = p.W.d;
    a.prod[j].y = p.y;
    a.prod[j].rows = p.W.rows;
  }
  a.nproducts = nproducts;
  a.x = x;
  a.nb = n / MLQ_QK;
  a.xq_out = xq_out;
  a.xd_out = xd_out;
  a.total_rows = 0;
  a.nchunks = 1;
  if ((flags & ~static_cast<unsigned>(MLQ_F_STATIC_WEIGHTS)) != 0) return MLQ_E_SHAPE;
  a.early = (flags & MLQ_F_STATIC_WEIGHTS) ? 1 : 0;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  if (!ctx.pdl) a.early = 0;  // without dependent launch there is nothing to overlap
  return from_cuda(mlq::launch_matvec_fused(ctx, type, a));
}

static_assert(MLQ_FUSED_MAX_PRODUCTS == mlq::kFusedMaxProducts, "header and kernels agree");
static_assert(MLQ_PHASE_MAX_PREFETCH == mlq::kPhaseMaxPrefetch, "header and kernels agree");

mlq_status mlq_decode_phase(const mlq_phase_input *in, const mlq_phase_product *products,
                            int nproducts, const void *const *prefetch,
                            const size_t *prefetch_bytes, int nprefetch, unsigned flags,
                            void *stream) {
  mlq::diag_entry("mlq_decode_phase", "n=%d products=%d input=%s", in ? in->n : -1, nproducts, in && in->x ? "f32" : "q8");
  if (in == nullptr || products == nullptr) return MLQ_E_NULL;
  if (nprefetch < 0 || nprefetch > MLQ_PHASE_MAX_PREFETCH) return MLQ_E_SHAPE;
  if (nprefetch > 0 && (prefetch == nullptr || prefetch_bytes == nullptr)) return MLQ_E_NULL;
  const int n = in->n;
  if (in->x != nullptr) {
    if (in->xq != nullptr || in->xd != nullptr) return MLQ_E_SHAPE;  // one input, not two
    if ((in->xq_out == nullptr) != (in->xd_out == nullptr)) return MLQ_E_NULL;
  } else {
    if (in->xq == nullptr || in->xd == nullptr) return MLQ_E_NULL;
    if (in->xq_out != nullptr || in->xd_out != nullptr) return MLQ_E_SHAPE;
  }
  if (nproducts < 1 || nproducts > MLQ_FUSED_MAX_PRODUCTS || !cols_ok(n)) return MLQ_E_SHAPE;
  if (!aligned(in->x, 16) || !aligned(in->xq, 16) || !aligned(in->xd, 16) ||
      !aligned(in->xq_out, 16) || !aligned(in->xd_out, 16))
    return MLQ_E_ALIGN;
  if ((flags & ~static_cast<unsigned>(MLQ_F_STATIC_WEIGHTS | MLQ_F_STATIC_INPUT)) != 0) return MLQ_E_SHAPE;
  mlq::FusedArgs a = {};
  const uint8_t type = products[0].W.type;
  bool any_yq = false;
  for (int j = 0; j < nproducts; ++j) {
    const mlq_phase_product &p = products[j];
    if (p.W.type != MLQ_Q4_0 && p.W.type != MLQ_Q8_0) return MLQ_E_TYPE;
    if (p.W.type != type) return MLQ_E_TYPE;
    if (p.W.cols != n || p.W.rows < 0) return MLQ_E_SHAPE;
    if ((p.yq == nullptr) != (p.yd == nullptr)) return MLQ_E_NULL;
    if (p.W.rows > 0 && (p.W.q == nullptr || p.W.d == nullptr || p.y == nullptr)) return MLQ_E_NULL;
    if (!aligned(p.W.q, 16) || !aligned(p.W.d, 16) || !aligned(p.y, 4) || !aligned(p.yq, 16) ||
        !aligned(p.yd, 16))
      return MLQ_E_ALIGN;
    any_yq = any_yq || p.yq != nullptr;
    a.prod[j].wq = static_cast<const uint8_t *>(p.W.q);
    a.prod[j].wd = p.W.d;
    a.prod[j].y = p.y;
    a.prod[j].rows = p.W.rows;
    a.prod[j].yq = p.yq;
    a.prod[j].yd = p.yd;
  }
  if (any_yq) {
    for (int j = 0; j < nproducts; ++j)
      if (products[j].W.rows % MLQ_QK != 0) return MLQ_E_SHAPE;
  }
  a.nproducts = nproducts;
  a.x = in->x;
  a.xq_in = in->xq;
  a.xd_in = in->xd;
  a.nb = n / MLQ_QK;
  a.xq_out = in->xq_out;
  a.xd_out = in->xd_out;
  a.any_yq = any_yq ? 1 : 0;
  a.nchunks = 1;
  a.early = (flags & MLQ_F_STATIC_WEIGHTS) ? 1 : 0;
  a.early_input = (flags & MLQ_F_STATIC_INPUT) && in->x != nullptr ? 1 : 0;
  for (int i = 0; i < nprefetch; ++i) {
    if (prefetch_bytes[i] > 0 && prefetch[i] == nullptr) return MLQ_E_NULL;
    a.pf_ptr[a.npf] = prefetch[i];
    a.pf_bytes[a.npf] = prefetch_bytes[i];
    a.npf += prefetch_bytes[i] > 0 ? 1 : 0;
  }
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  if (!ctx.pdl) a.early = a.early_input = 0;  // without dependent launch there is nothing to overlap
  return from_cuda(mlq::launch_matvec_fused(ctx, type, a));
}

size_t mlq_chain_workspace_bytes(int nphases) {
  return nphases < 0 ? 0 : static_cast<size_t>(nphases + 1) * sizeof(unsigned);
}

mlq_status mlq_decode_chain(const mlq_chain_phase *phases, int nphases,
                            const mlq_chain_product *products, int nproducts, void *workspace,
                            size_t workspace_bytes, void *stream) {
  mlq::diag_entry("mlq_decode_chain", "phases=%d products=%d", nphases, nproducts);
  mlq::ChainArgs a;
  mlq_status s = build_chain_args(phases, nphases, products, nproducts, &a);
  if (s != MLQ_OK) return s;
  if (workspace == nullptr) return MLQ_E_NULL;
  if (!aligned(workspace, 4)) return MLQ_E_ALIGN;
  if (workspace_bytes < mlq_chain_workspace_bytes(nphases)) return MLQ_E_SHAPE;
  a.counters = static_cast<unsigned *>(workspace);
  mlq::LaunchCtx ctx;
  s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_decode_chain(ctx, products[0].W.type, a));
}

// The fixed counter array holds one word per phase plus the exit counter.
static_assert(MLQ_CHAIN_STATIC_MAX_PHASES + 1 <= mlq::kStaticChainWords,
              "the static chain's counter array is too small for its phase limit");

mlq_status mlq_decode_chain_static(const mlq_chain_phase *phases, int nphases,
                                   const mlq_chain_product *products, int nproducts,
                                   void *stream) {
  mlq::diag_entry("mlq_decode_chain_static", "phases=%d products=%d", nphases, nproducts);
  mlq::ChainArgs a;
  mlq_status s = build_chain_args(phases, nphases, products, nproducts, &a);
  if (s != MLQ_OK) return s;
  if (nphases > MLQ_CHAIN_STATIC_MAX_PHASES) return MLQ_E_SHAPE;
  mlq::LaunchCtx ctx;
  s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MLQ_E_CUDA;
  }
  return from_cuda(mlq::launch_decode_chain_static(ctx, dev, products[0].W.type, a));
}

mlq_status mlq_debug_chain_plan(const mlq_chain_phase *phases, int nphases,
                                const mlq_chain_product *products, int nproducts, int num_sms,
                                int32_t *info, int info_len) {
  mlq::ChainArgs a;
  mlq_status s = build_chain_args(phases, nphases, products, nproducts, &a);
  if (s != MLQ_OK) return s;
  if (info == nullptr) return MLQ_E_NULL;
  if (num_sms < 1 || info_len < 0) return MLQ_E_SHAPE;
  return mlq::describe_decode_stream(num_sms, products[0].W.type, a, info, info_len) < 0 ? MLQ_E_SHAPE
                                                                                          : MLQ_OK;
}

mlq_status mlq_prefetch_l2(const void *const *ptrs, const size_t *bytes, int n, void *stream) {
  mlq::diag_entry("mlq_prefetch_l2", "");
  if (n < 0 || n > MLQ_MAX_PREFETCH_RANGES) return MLQ_E_SHAPE;
  if (n > 0 && (ptrs == nullptr || bytes == nullptr)) return MLQ_E_NULL;
  mlq::PrefetchList list;
  list.n = n;
  for (int i = 0; i < n; ++i) {
    if (ptrs[i] == nullptr && bytes[i] != 0) return MLQ_E_NULL;
    list.ptr[i] = ptrs[i];
    list.bytes[i] = bytes[i];
  }
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_prefetch_l2(ctx, list));
}

// ---- Q4_K-style super-blocks ---------------------------------------------------
namespace {
bool q4k_cols_ok(int cols) { return cols > 0 && cols % 256 == 0 && cols <= MLQ_MAX_COLS; }

mlq_status check_q4k(const mlq_q4k_tensor *W, const mlq_q8k_act *x, int r0, int r1) {
  if (W == nullptr || x == nullptr) return MLQ_E_NULL;
  if (W->q == nullptr || W->s == nullptr || W->d == nullptr || W->dmin == nullptr) return MLQ_E_NULL;
  if (x->q == nullptr || x->d == nullptr || x->bsums == nullptr) return MLQ_E_NULL;
  if (!q4k_cols_ok(W->cols) || W->rows < 0 || x->n != W->cols) return MLQ_E_SHAPE;
  if (r0 < 0 || r1 < r0 || r1 > W->rows) return MLQ_E_SHAPE;
  if (!aligned(W->q, 16) || !aligned(W->s, 16) || !aligned(W->d, 4) || !aligned(W->dmin, 4))
    return MLQ_E_ALIGN;
  if (!aligned(x->q, 16) || !aligned(x->d, 16) || !aligned(x->bsums, 16)) return MLQ_E_ALIGN;
  return MLQ_OK;
}

mlq_status q4k_common(float *y, int32_t *isum, int32_t *msum, const mlq_q4k_tensor *W,
                      const mlq_q8k_act *x, int r0, int r1, void *stream) {
  mlq_status s = check_q4k(W, x, r0, r1);
  if (s != MLQ_OK) return s;
  if (y != nullptr && !aligned(y, 4)) return MLQ_E_ALIGN;
  if (isum != nullptr && (!aligned(isum, 4) || !aligned(msum, 4))) return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  if ((s = make_ctx(&ctx, stream)) != MLQ_OK) return s;
  return from_cuda(mlq::launch_matvec_q4k(ctx, W->q, W->s, W->d, W->dmin, W->cols / 256, x->q, x->d,
                                          x->bsums, y, isum, msum, r0, r1));
}
}  // namespace

mlq_status mlq_quantize_q8k(mlq_q8k_act *out, const float *x, int k, void *stream) {
  mlq::diag_entry("mlq_quantize_q8k", "k=%d", k);
  if (out == nullptr || x == nullptr || out->q == nullptr || out->d == nullptr || out->bsums == nullptr)
    return MLQ_E_NULL;
  if (!q4k_cols_ok(k) || out->n != k) return MLQ_E_SHAPE;
  if (!aligned(x, 16) || !aligned(out->q, 16) || !aligned(out->d, 16) || !aligned(out->bsums, 16))
    return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_quantize_q8k(ctx, x, out->q, out->d, out->bsums, k));
}

mlq_status mlq_matvec_q4k(float *y, const mlq_q4k_tensor *W, const mlq_q8k_act *x, int r0, int r1,
                          void *stream) {
  mlq::diag_entry("mlq_matvec_q4k", "rows=%d cols=%d r=[%d,%d)", W ? W->rows : -1, W ? W->cols : -1, r0, r1);
  if (y == nullptr) return MLQ_E_NULL;
  return q4k_common(y, nullptr, nullptr, W, x, r0, r1, stream);
}

mlq_status mlq_block_sums_q4k(int32_t *isum, int32_t *msum, const mlq_q4k_tensor *W,
                              const mlq_q8k_act *x, int r0, int r1, void *stream) {
  if (isum == nullptr || msum == nullptr) return MLQ_E_NULL;
  return q4k_common(nullptr, isum, msum, W, x, r0, r1, stream);
}

mlq_status mlq_q4k_phase(const float *x, int k, const mlq_q4k_product *products, int nproducts,
                         unsigned flags, void *stream) {
  mlq::diag_entry("mlq_q4k_phase", "k=%d products=%d flags=%u", k, nproducts, flags);
  if (x == nullptr || products == nullptr) return MLQ_E_NULL;
  if (nproducts < 1 || nproducts > 4 || !q4k_cols_ok(k)) return MLQ_E_SHAPE;
  if ((flags & ~MLQ_F_STATIC_INPUT) != 0) return MLQ_E_SHAPE;
  if (!aligned(x, 16)) return MLQ_E_ALIGN;
  mlq::Q4KProductDev p[4];
  for (int j = 0; j < nproducts; ++j) {
    const mlq_q4k_tensor &W = products[j].W;
    if (products[j].y == nullptr || W.q == nullptr || W.s == nullptr || W.d == nullptr ||
        W.dmin == nullptr)
      return MLQ_E_NULL;
    if (W.cols != k || W.rows < 0) return MLQ_E_SHAPE;
    if (!aligned(W.q, 16) || !aligned(W.s, 16) || !aligned(W.d, 4) || !aligned(W.dmin, 4) ||
        !aligned(products[j].y, 4))
      return MLQ_E_ALIGN;
    p[j] = mlq::Q4KProductDev{W.q, W.s, W.d, W.dmin, products[j].y, W.rows};
  }
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_phase_q4k(ctx, x, k / 256, p, nproducts,
                                         ctx.pdl && (flags & MLQ_F_STATIC_INPUT) != 0));
}

// ---- block length 32 / 128, float16 scales, signed-offset 8-bit ---------------
namespace {
mlq_status check_nbits(const mlq_nbits_tensor *W, const mlq_blk_act *x, int r0, int r1) {
  if (W == nullptr || x == nullptr) return MLQ_E_NULL;
  if (W->q == nullptr || W->scales == nullptr || x->q == nullptr || x->d == nullptr || x->bsums == nullptr)
    return MLQ_E_NULL;
  if (W->bits != 4 && W->bits != 8) return MLQ_E_TYPE;
  if (W->scale_f16 != 0 && W->scale_f16 != 1) return MLQ_E_TYPE;
  if (W->bits == 4 && W->zp != nullptr) return MLQ_E_TYPE;
  if (W->blk != 32 && W->blk != 128) return MLQ_E_SHAPE;
  if (W->cols <= 0 || W->cols % W->blk != 0 || W->cols > MLQ_MAX_COLS || W->rows < 0) return MLQ_E_SHAPE;
  if (x->n != W->cols || x->blk != W->blk) return MLQ_E_SHAPE;
  if (r0 < 0 || r1 < r0 || r1 > W->rows) return MLQ_E_SHAPE;
  const int nb = W->cols / W->blk;
  if (W->scale_ld < nb || (W->scale_ld * (W->scale_f16 ? 2 : 4)) % 16 != 0) return MLQ_E_SHAPE;
  if (W->zp != nullptr && (W->zp_ld < nb || W->zp_ld % 16 != 0)) return MLQ_E_SHAPE;
  if (!aligned(W->q, 16) || !aligned(W->scales, 16) || !aligned(W->zp, 16)) return MLQ_E_ALIGN;
  if (!aligned(x->q, 16) || !aligned(x->d, 4) || !aligned(x->bsums, 4)) return MLQ_E_ALIGN;
  return MLQ_OK;
}

mlq_status nbits_common(float *y, int32_t *sumi, const mlq_nbits_tensor *W, const mlq_blk_act *x,
                        int r0, int r1, void *stream) {
  mlq_status s = check_nbits(W, x, r0, r1);
  if (s != MLQ_OK) return s;
  if (!aligned(y != nullptr ? static_cast<const void *>(y) : static_cast<const void *>(sumi), 4))
    return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  if ((s = make_ctx(&ctx, stream)) != MLQ_OK) return s;
  return from_cuda(mlq::launch_matvec_nbits(ctx, W->bits, W->blk, W->q, W->scales, W->scale_f16,
                                            W->scale_ld, W->zp, W->zp_ld, W->cols, x->q, x->d,
                                            x->bsums, y, sumi, r0, r1));
}
}  // namespace

mlq_status mlq_quantize_blk(mlq_blk_act *out, const float *x, int k, void *stream) {
  mlq::diag_entry("mlq_quantize_blk", "k=%d blk=%d", k, out ? out->blk : -1);
  if (out == nullptr || x == nullptr || out->q == nullptr || out->d == nullptr || out->bsums == nullptr)
    return MLQ_E_NULL;
  if (out->blk != 32 && out->blk != 128) return MLQ_E_SHAPE;
  if (k <= 0 || k % out->blk != 0 || k > MLQ_MAX_COLS || out->n != k) return MLQ_E_SHAPE;
  if (!aligned(x, 16) || !aligned(out->q, 16) || !aligned(out->d, 4) || !aligned(out->bsums, 4))
    return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_quantize_blk(ctx, x, out->q, out->d, out->bsums, k, out->blk));
}

mlq_status mlq_nbits_phase(const float *x, int k, const mlq_nbits_product *products, int nproducts,
                           unsigned flags, void *stream) {
  mlq::diag_entry("mlq_nbits_phase", "k=%d products=%d flags=%u", k, nproducts, flags);
  if (x == nullptr || products == nullptr) return MLQ_E_NULL;
  if (nproducts < 1 || nproducts > 4) return MLQ_E_SHAPE;
  if ((flags & ~MLQ_F_STATIC_INPUT) != 0) return MLQ_E_SHAPE;
  if (!aligned(x, 16)) return MLQ_E_ALIGN;
  const mlq_nbits_tensor &W0 = products[0].W;
  mlq::NBitsProductDev p[4];
  for (int j = 0; j < nproducts; ++j) {
    const mlq_nbits_tensor &W = products[j].W;
    if (products[j].y == nullptr || W.q == nullptr || W.scales == nullptr) return MLQ_E_NULL;
    if (W.bits != 4 && W.bits != 8) return MLQ_E_TYPE;
    if (W.scale_f16 != 0 && W.scale_f16 != 1) return MLQ_E_TYPE;
    if (W.bits == 4 && W.zp != nullptr) return MLQ_E_TYPE;
    // one format and one row layout of scales and zero points for all
    if (W.bits != W0.bits || W.scale_f16 != W0.scale_f16 || (W.zp == nullptr) != (W0.zp == nullptr))
      return MLQ_E_TYPE;
    if (W.blk != W0.blk || W.scale_ld != W0.scale_ld || (W.zp != nullptr && W.zp_ld != W0.zp_ld))
      return MLQ_E_SHAPE;
    if (W.blk != 32 && W.blk != 128) return MLQ_E_SHAPE;
    if (W.cols != k || k <= 0 || k % W.blk != 0 || k > MLQ_MAX_COLS || W.rows < 0) return MLQ_E_SHAPE;
    const int nb = k / W.blk;
    if (W.scale_ld < nb || (W.scale_ld * (W.scale_f16 ? 2 : 4)) % 16 != 0) return MLQ_E_SHAPE;
    if (W.zp != nullptr && (W.zp_ld < nb || W.zp_ld % 16 != 0)) return MLQ_E_SHAPE;
    if (!aligned(W.q, 16) || !aligned(W.scales, 16) || !aligned(W.zp, 16) || !aligned(products[j].y, 4))
      return MLQ_E_ALIGN;
    p[j] = mlq::NBitsProductDev{W.q, W.scales, W.zp, products[j].y, W.rows};
  }
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_phase_nbits(ctx, W0.bits, W0.blk, W0.scale_f16, W0.scale_ld, W0.zp_ld, k,
                                           x, p, nproducts, ctx.pdl && (flags & MLQ_F_STATIC_INPUT) != 0));
}

mlq_status mlq_matvec_nbits(float *y, const mlq_nbits_tensor *W, const mlq_blk_act *x, int r0, int r1,
                            void *stream) {
  mlq::diag_entry("mlq_matvec_nbits", "rows=%d cols=%d bits=%d blk=%d r=[%d,%d)", W ? W->rows : -1, W ? W->cols : -1, W ? W->bits : -1, W ? W->blk : -1, r0, r1);
  if (y == nullptr) return MLQ_E_NULL;
  return nbits_common(y, nullptr, W, x, r0, r1, stream);
}

mlq_status mlq_block_sumi_nbits(int32_t *sumi, const mlq_nbits_tensor *W, const mlq_blk_act *x, int r0,
                                int r1, void *stream) {
  if (sumi == nullptr) return MLQ_E_NULL;
  return nbits_common(nullptr, sumi, W, x, r0, r1, stream);
}

// ---- the floating-point steps of a decode layer -------------------------------
namespace {
// An optional Q8_0 output of n elements (one row): both arrays or none.
mlq_status check_q8_out(const mlq_qact *o, int n) {
  if (o == nullptr) return MLQ_OK;
  if (o->q == nullptr || o->d == nullptr) return MLQ_E_NULL;
  if (!cols_ok(n) || o->n != n || o->m != 1) return MLQ_E_SHAPE;
  if (!aligned(o->q, 16) || !aligned(o->d, 16)) return MLQ_E_ALIGN;
  return MLQ_OK;
}
bool floats_ok(const void *p) { return aligned(p, 4); }
}  // namespace

mlq_status mlq_rmsnorm(float *o, const float *x, const float *w, int n, float eps, mlq_qact *oq,
                       void *stream) {
  mlq::diag_entry("mlq_rmsnorm", "n=%d", n);
  if (x == nullptr || w == nullptr || (o == nullptr && oq == nullptr)) return MLQ_E_NULL;
  if (n < 1 || n > MLQ_MAX_COLS || !(eps >= 0.0f)) return MLQ_E_SHAPE;
  if (!floats_ok(x) || !floats_ok(w) || !floats_ok(o)) return MLQ_E_ALIGN;
  mlq_status s = check_q8_out(oq, n);
  if (s != MLQ_OK) return s;
  mlq::LaunchCtx ctx;
  if ((s = make_ctx(&ctx, stream)) != MLQ_OK) return s;
  return from_cuda(mlq::launch_rmsnorm_q8(ctx, const_cast<float *>(x), nullptr, w, o,
                                          oq ? oq->q : nullptr, oq ? oq->d : nullptr, n, eps));
}

mlq_status mlq_add_rmsnorm(float *x, const float *y, const float *w, int n, float eps, float *o,
                           mlq_qact *oq, void *stream) {
  mlq::diag_entry("mlq_add_rmsnorm", "n=%d", n);
  if (x == nullptr || y == nullptr || w == nullptr || (o == nullptr && oq == nullptr)) return MLQ_E_NULL;
  if (n < 1 || n > MLQ_MAX_COLS || !(eps >= 0.0f)) return MLQ_E_SHAPE;
  if (!floats_ok(x) || !floats_ok(y) || !floats_ok(w) || !floats_ok(o)) return MLQ_E_ALIGN;
  mlq_status s = check_q8_out(oq, n);
  if (s != MLQ_OK) return s;
  mlq::LaunchCtx ctx;
  if ((s = make_ctx(&ctx, stream)) != MLQ_OK) return s;
  return from_cuda(mlq::launch_rmsnorm_q8(ctx, x, y, w, o, oq ? oq->q : nullptr,
                                          oq ? oq->d : nullptr, n, eps));
}

mlq_status mlq_add(float *y, const float *x, int n, void *stream) {
  mlq::diag_entry("mlq_add", "n=%d", n);
  if (y == nullptr || x == nullptr) return MLQ_E_NULL;
  if (n < 1 || n > MLQ_MAX_COLS) return MLQ_E_SHAPE;
  if (!floats_ok(y) || !floats_ok(x)) return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_add(ctx, y, x, n));
}

mlq_status mlq_softmax(float *x, int n, void *stream) {
  mlq::diag_entry("mlq_softmax", "n=%d", n);
  if (x == nullptr) return MLQ_E_NULL;
  if (n < 1 || n > MLQ_MAX_COLS) return MLQ_E_SHAPE;
  if (!floats_ok(x)) return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_softmax(ctx, x, n));
}

mlq_status mlq_silu_mul(float *g, const float *u, int n, mlq_qact *gq, void *stream) {
  mlq::diag_entry("mlq_silu_mul", "n=%d", n);
  if (g == nullptr || u == nullptr) return MLQ_E_NULL;
  if (n < 1 || n > MLQ_MAX_COLS) return MLQ_E_SHAPE;
  if (!floats_ok(g) || !floats_ok(u)) return MLQ_E_ALIGN;
  mlq_status s = check_q8_out(gq, n);
  if (s != MLQ_OK) return s;
  mlq::LaunchCtx ctx;
  if ((s = make_ctx(&ctx, stream)) != MLQ_OK) return s;
  return from_cuda(mlq::launch_silu_mul_q8(ctx, g, u, n, gq ? gq->q : nullptr, gq ? gq->d : nullptr));
}

mlq_status mlq_rope_tables(float *cos_t, float *sin_t, int max_seq, int head_dim, float theta,
                           void *stream) {
  mlq::diag_entry("mlq_rope_tables", "");
  if (cos_t == nullptr || sin_t == nullptr) return MLQ_E_NULL;
  if (max_seq < 1 || max_seq > MLQ_MAX_SEQ || head_dim < 2 || head_dim > MLQ_MAX_HEAD_DIM ||
      head_dim % 2 != 0 || !(theta > 0.0f))
    return MLQ_E_SHAPE;
  if (!floats_ok(cos_t) || !floats_ok(sin_t)) return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_rope_tables(ctx, cos_t, sin_t, max_seq, head_dim, theta));
}

namespace {
bool heads_ok(int head_dim, int n_heads, int n_kv_heads) {
  return head_dim >= 2 && head_dim <= MLQ_MAX_HEAD_DIM && head_dim % 2 == 0 && n_heads >= 1 &&
         n_kv_heads >= 1 && n_heads % n_kv_heads == 0 &&
         static_cast<long long>(n_heads) * head_dim <= MLQ_MAX_COLS;
}
}  // namespace

mlq_status mlq_rope(float *q, float *k, const float *cos_row, const float *sin_row, int head_dim,
                    int n_heads, int n_kv_heads, float *k_out, const float *v, float *v_out,
                    void *stream) {
  mlq::diag_entry("mlq_rope", "");
  if (q == nullptr || k == nullptr || cos_row == nullptr || sin_row == nullptr) return MLQ_E_NULL;
  if ((v == nullptr) != (v_out == nullptr)) return MLQ_E_NULL;
  if (!heads_ok(head_dim, n_heads, n_kv_heads)) return MLQ_E_SHAPE;
  if (!floats_ok(q) || !floats_ok(k) || !floats_ok(cos_row) || !floats_ok(sin_row) ||
      !floats_ok(k_out) || !floats_ok(v) || !floats_ok(v_out))
    return MLQ_E_ALIGN;
  mlq::LaunchCtx ctx;
  mlq_status s = make_ctx(&ctx, stream);
  if (s != MLQ_OK) return s;
  return from_cuda(mlq::launch_rope_call(ctx, q, k, k_out, v, v_out, cos_row, sin_row, head_dim,
                                         n_heads, n_kv_heads));
}

mlq_status mlq_attention(float *o, mlq_qact *oq, const float *q, const float *k_cache,
                         const float *v_cache, int n_pos, int head_dim, int n_heads, int n_kv_heads,
                         void *stream) {
  mlq::diag_entry("mlq_attention", "");
  if (o == nullptr || q == nullptr || k_cache == nullptr || v_cache == nullptr) return MLQ_E_NULL;
  if (!heads_ok(head_dim, n_heads, n_kv_heads) || n_pos < 1 || n_pos > MLQ_MAX_SEQ) return MLQ_E_SHAPE;
  if (oq != nullptr && head_dim % MLQ_QK != 0) return MLQ_E_SHAPE;
  if (!floats_ok(o) || !floats_ok(q) || !floats_ok(k_cache) || !floats_ok(v_cache)) return MLQ_E_ALIGN;
  mlq_status s = check_q8_out(oq, n_heads * head_dim);
  if (s != MLQ_OK) return s;
  mlq::LaunchCtx ctx;
  if ((s = make_ctx(&ctx, stream)) != MLQ_OK) return s;
  return from_cuda(mlq::launch_attention_call(ctx, o, oq ? oq->q : nullptr, oq ? oq->d : nullptr, q,
                                              k_cache, v_cache, n_pos, head_dim, n_heads,
                                              n_kv_heads));
}

mlq_status mlq_last_device_error(void *stream) {
  DevInfo *d = nullptr;
  mlq_status s = device_info(&d);
  if (s != MLQ_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLQ_E_CUDA;
  }
  int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MLQ_E_CUDA;
  }
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return MLQ_E_CUDA;
    }
    return static_cast<mlq_status>(v);
  }
  return MLQ_OK;
}

mlq_status mlq_debug_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_ns.store(limit_ns, std::memory_order_relaxed);
  return MLQ_OK;
}

const char *mlq_status_str(mlq_status s) {
  switch (s) {
    case MLQ_OK: return "MLQ_OK";
    case MLQ_E_SHAPE: return "MLQ_E_SHAPE";
    case MLQ_E_ALIGN: return "MLQ_E_ALIGN";
    case MLQ_E_TYPE: return "MLQ_E_TYPE";
    case MLQ_E_NULL: return "MLQ_E_NULL";
    case MLQ_E_ARCH: return "MLQ_E_ARCH";
    case MLQ_E_CUDA: return "MLQ_E_CUDA";
    case MLQ_E_TIMEOUT: return "MLQ_E_TIMEOUT";
    case MLQ_E_BOUNDS: return "MLQ_E_BOUNDS";
  }
  return "MLQ_E_UNKNOWN";
}

}  // extern "C"
