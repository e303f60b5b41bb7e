// qmv_api.cu -- the C ABI of libqmv (declared in include/qmv.h): argument checks, the
// layout of a matrix image, kernel selection and the per-device status word.
//
// Layout (Krafla ".mlb model format v1", "Body"): q array, zero padding to a multiple of 64
// bytes, d array.  Checks follow the loader's classes ("Validation done by the loader"):
// unknown enum -> format error; zero dimension, cols not a multiple of 32, overflow -> shape.
#include <mutex>

#include "qmv_common.cuh"
#include "qmv_internal.h"

namespace qmv {

// The per-device status word (one copy per device that loads the library).
__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kPrefillMinBatch = 17;  // from here on the prefill kernel takes bf16 batches
constexpr int kTcMinBatch = 8;        // bf16 passes of this many vectors may go to decode_tc:
constexpr long long kTcMinBytes = 128LL << 20;     // launches of this many weight bytes (below, and at
                                                   // 2..7 vectors, the mma.sync kernel measured faster)
constexpr long long kTcWideMinBytes = 8LL << 20;   // passes of 9..16 vectors in one decode_tc launch
constexpr long long kTcF32MinBytes = 96LL << 20;   // float32 passes of 2..8 vectors take decode_tc from here
constexpr long long kQxBdiagMaxBytes = 96LL << 20;  // one-vector activation-quantized groups below this
                                                    // size take the block-diagonal kernel
constexpr long long kF32SplitMinWeights = 256LL << 10;  // one f32 vector: split hi/lo from this many weights
// one f32 vector: split in the product's own activation stage (one launch) below this many
// weight bytes; above it the split kernel runs once per column and the product reads its parts
// (every row tile of a large launch redoing the split measured 25% more instructions per stage)
constexpr long long kF32InKernelMaxBytes = 16LL << 20;
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};

struct Layout {
  int64_t q_bytes, d_off, d_bytes;
};

int make_layout(int wtype, int scale_dtype, int64_t rows, int64_t cols, Layout* L) {
  if (wtype != QMV_Q8_0 && wtype != QMV_Q4_0) return QMV_E_FORMAT;
  if (scale_dtype != QMV_SCALE_F32 && scale_dtype != QMV_SCALE_F16) return QMV_E_FORMAT;
  if (rows <= 0 || cols <= 0 || cols % 32 != 0) return QMV_E_SHAPE;
  if (rows > INT64_MAX / cols) return QMV_E_SHAPE;
  const int64_t n = rows * cols;
  if (n > INT64_MAX / 4) return QMV_E_SHAPE;
  L->q_bytes = (wtype == QMV_Q8_0) ? n : n / 2;
  L->d_bytes = (n / 32) * (scale_dtype == QMV_SCALE_F16 ? 2 : 4);
  L->d_off = (L->q_bytes + 63) / 64 * 64;
  if (L->d_off > INT64_MAX - L->d_bytes) return QMV_E_SHAPE;
  return QMV_OK;
}

int make_ref(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void* W, MatrixRef* m) {
  Layout L;
  const int st = make_layout(wtype, scale_dtype, rows, cols, &L);
  if (st != QMV_OK) return st;
  if (W == nullptr) return QMV_E_ARG;
  if (reinterpret_cast<uintptr_t>(W) % 16 != 0) return QMV_E_ALIGN;
  m->wtype = wtype;
  m->scale_f16 = scale_dtype == QMV_SCALE_F16;
  m->rows = rows;
  m->cols = cols;
  m->q = static_cast<const uint8_t*>(W);
  m->d = m->q + L.d_off;
  return QMV_OK;
}

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

cudaError_t current_device_info(DeviceInfo* info) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev_ready[dev]) {
    DeviceInfo d{};
    d.device = dev;
    if ((err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return err;
    int optin = 0;
    if ((err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return err;
    d.smem_optin = (size_t)optin;
    int per_sm = 0, reserved = 0;
    if ((err = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
      return err;
    if ((err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
      return err;
    d.smem_per_sm = (size_t)per_sm;
    d.smem_reserved = (size_t)reserved;
    void* sym = nullptr;
    if ((err = cudaGetSymbolAddress(&sym, g_device_status)) != cudaSuccess) return err;
    d.status = static_cast<int*>(sym);
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
  }
  *info = g_dev[dev];
  return cudaSuccess;
}

}  // namespace qmv

using namespace qmv;

// Scratch of qmv_matvec_grouped_noalloc: split-tile arrival counters and partial sums of
// the tensor-memory decode kernel for up to QMV_NOALLOC_MAX_CTAS CTAs, in the layout of a
// per-stream workspace.  Zero-initialized when this module is loaded onto a device (on the
// library's first call that needs it there: modules load lazily).  A launch that completes
// leaves the counters at zero (the last arrival at a split tile resets its counter); after a
// kernel gave up on a bounded wait, qmv_check_device() clears them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QMV_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};
}  // namespace

// Device address of g_noalloc_scratch on `device` (the current device), looked up once.
static cudaError_t noalloc_scratch(int device, void** base) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[device] == nullptr) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_noalloc_addr[device] = p;
  }
  *base = g_noalloc_addr[device];
  return cudaSuccess;
}

// Zero the arrival counters of g_noalloc_scratch on `device` (the current device) if the
// entry point has been used there; synchronous.
static cudaError_t noalloc_reset(int device) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[device] == nullptr) return cudaSuccess;
  Workspace ws;
  workspace_carve(g_noalloc_addr[device], sizeof(g_noalloc_scratch), QMV_NOALLOC_MAX_CTAS, &ws);
  return cudaMemset(ws.counters, 0, workspace_counter_bytes(ws.max_counters));
}

extern "C" {

size_t qmv_weight_bytes(int wtype, int scale_dtype, int64_t rows, int64_t cols) {
  Layout L;
  if (make_layout(wtype, scale_dtype, rows, cols, &L) != QMV_OK) return 0;
  return (size_t)(L.d_off + L.d_bytes);
}

int64_t qmv_scale_offset(int wtype, int scale_dtype, int64_t rows, int64_t cols) {
  Layout L;
  if (make_layout(wtype, scale_dtype, rows, cols, &L) != QMV_OK) return -1;
  return L.d_off;
}

int qmv_matrix_wtype(int file_wtype, uint32_t q8_mask, int class_bit, int shared_classifier) {
  if (file_wtype != QMV_Q8_0 && file_wtype != QMV_Q4_0) return -1;
  switch (class_bit) {
    case QMV_CLASS_TOK_EMB: case QMV_CLASS_WCLS: case QMV_CLASS_WQ_WK: case QMV_CLASS_WV:
    case QMV_CLASS_WO: case QMV_CLASS_W1_W3: case QMV_CLASS_W2: break;
    default: return -1;
  }
  if (file_wtype == QMV_Q8_0) return QMV_Q8_0;
  uint32_t bits = (uint32_t)class_bit;
  if (class_bit == QMV_CLASS_TOK_EMB && shared_classifier) bits |= QMV_CLASS_WCLS;
  return (q8_mask & bits) ? QMV_Q8_0 : QMV_Q4_0;
}

int qmv_matvec_grouped(int wtype, int scale_dtype, int x_dtype, int batch, const qmv_problem* problems, int n,
                       unsigned flags, cudaStream_t stream) {
  if (problems == nullptr || n < 1 || n > QMV_MAX_GROUP) return QMV_E_ARG;
  if (x_dtype != QMV_X_F32 && x_dtype != QMV_X_BF16 && x_dtype != QMV_X_SILU_GLU_F32 &&
      x_dtype != QMV_X_GELU_GLU_F32 && x_dtype != QMV_X_BF16_PAIR)
    return QMV_E_FORMAT;
  if (batch < 0) return QMV_E_ARG;
  if ((flags & ~(QMV_FLAG_OVERLAP | QMV_FLAG_BF16_WEIGHTS)) != 0) return QMV_E_ARG;
  const bool pair = x_dtype == QMV_X_BF16_PAIR;
  if (pair && batch > 1) return QMV_E_ARG;
  // gated activations: x holds gate then up (batch x cols float32 each); act(gate) * up is
  // formed in the activation prep of the float32 routes
  const bool glu = x_dtype == QMV_X_SILU_GLU_F32 || x_dtype == QMV_X_GELU_GLU_F32;
  const int act = x_dtype == QMV_X_SILU_GLU_F32 ? 0 : x_dtype == QMV_X_GELU_GLU_F32 ? 1 : -1;
  MatrixRef ms[QMV_MAX_GROUP];
  for (int i = 0; i < n; ++i) {
    const qmv_problem& pr = problems[i];
    const int st = make_ref(wtype, scale_dtype, pr.rows, pr.cols, pr.W, &ms[i]);
    if (st != QMV_OK) return st;
    if (batch == 0) continue;
    if (pr.x == nullptr || pr.y == nullptr) return QMV_E_ARG;
    if (!aligned(pr.x, 16) || !aligned(pr.y, 4)) return QMV_E_ALIGN;
    if (pr.rows > INT64_MAX / batch) return QMV_E_SHAPE;
    if ((glu || pair) && !matvec_mma_supported(ms[i])) return QMV_E_SHAPE;
  }
  if (batch == 0) return QMV_OK;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  if (pair) {
    // one vector given as its bfloat16 hi and lo parts: the block-diagonal kernel runs every
    // block's MMAs once with each
    const void* xs[QMV_MAX_GROUP];
    float* ys[QMV_MAX_GROUP];
    for (int i = 0; i < n; ++i) {
      xs[i] = problems[i].x;
      ys[i] = problems[i].y;
    }
    return launch_matvec_bdiag_split(ms, xs, ys, n, (flags & QMV_FLAG_OVERLAP) != 0, dev, stream) == cudaSuccess
               ? QMV_OK
               : QMV_E_CUDA;
  }
  const bool xb = x_dtype == QMV_X_BF16;
  const size_t xsz = xb ? 2 : 4;
  const bool pdl = (flags & QMV_FLAG_OVERLAP) != 0;
  auto weight_bytes = [&](const MatrixRef& m) {
    return m.rows * m.cols / 32 * ((wtype == QMV_Q4_0 ? 16 : 32) + (scale_dtype == QMV_SCALE_F16 ? 2 : 4));
  };
  long long group_bytes = 0;
  for (int i = 0; i < n; ++i) group_bytes += weight_bytes(ms[i]);
  // 17 or more bf16 vectors (16 in groups under 8 MB of weights, where it measured faster
  // than one 16-vector pass of the tensor-memory decode kernel): the prefill kernel, per
  // problem, in passes of up to 128
  const bool prefill_batch = batch >= kPrefillMinBatch || (batch == 16 && group_bytes < kTcWideMinBytes);
  bool use_prefill[QMV_MAX_GROUP];
  bool any_decode = false;
  for (int i = 0; i < n; ++i) {
    use_prefill[i] = prefill_batch && prefill_supported(ms[i], xb);
    if (use_prefill[i]) {
      // split tiles between CTAs when the stream has its prefill workspace (created on the
      // stream's first prefill call, never while it is captured)
      Workspace pws;
      const Workspace* pw = stream_prefill_workspace(dev, stream, &pws) == cudaSuccess ? &pws : nullptr;
      const int pmax = prefill_max_batch();
      for (int b0 = 0; b0 < batch; b0 += pmax) {
        const int nb = (batch - b0) < pmax ? (batch - b0) : pmax;
        const void* xp = static_cast<const uint8_t*>(problems[i].x) + (size_t)b0 * (size_t)ms[i].cols * xsz;
        float* yp = problems[i].y + (size_t)b0 * (size_t)ms[i].rows;
        if (launch_prefill(ms[i], xp, yp, nb, (flags & QMV_FLAG_BF16_WEIGHTS) != 0, dev, pw, pdl, stream) !=
            cudaSuccess)
          return QMV_E_CUDA;
      }
    } else {
      any_decode = true;
    }
  }
  if (!any_decode) return QMV_OK;
  // problems the tensor-core kernel takes go in one launch per pass of 8 vectors; the rest
  // run the general kernel one by one.  bf16 batches of 9 or more whose problems the
  // tensor-memory kernel takes all, 8 MB of weights or more, on a stream with its workspace:
  // passes of 16 (that kernel's 16 MMA columns then all hold vectors)
  long long decode_bytes = 0;
  for (int i = 0; i < n; ++i)
    if (!use_prefill[i]) decode_bytes += weight_bytes(ms[i]);
  bool wide = xb && batch > 8 && decode_bytes >= kTcWideMinBytes;
  for (int i = 0; i < n && wide; ++i)
    wide = use_prefill[i] || (matvec_mma_supported(ms[i]) && decode_tc_supported(ms[i]));
  if (wide) {
    Workspace probe;
    wide = stream_workspace(dev, stream, &probe) == cudaSuccess;
  }
  const int pass = wide ? 16 : 8;
  MatrixRef fast[QMV_MAX_GROUP];
  const void* fx[QMV_MAX_GROUP];
  float* fy[QMV_MAX_GROUP];
  for (int b0 = 0; b0 < batch; b0 += pass) {
    const int nb = (batch - b0) < pass ? (batch - b0) : pass;
    int nf = 0;
    for (int i = 0; i < n; ++i) {
      if (use_prefill[i]) continue;
      const void* xp = static_cast<const uint8_t*>(problems[i].x) + (size_t)b0 * (size_t)ms[i].cols * xsz;
      float* yp = problems[i].y + (size_t)b0 * (size_t)ms[i].rows;
      if (matvec_mma_supported(ms[i])) {
        fast[nf] = ms[i];
        fx[nf] = xp;
        fy[nf] = yp;
        ++nf;
      } else if (launch_matvec_simple(ms[i], xp, xb, yp, nb, dev, stream) != cudaSuccess) {
        return QMV_E_CUDA;
      }
    }
    if (nf == 0) continue;
    // bf16 activations: the tensor-memory kernel for passes of 9..16 vectors and passes of 8
    // over 128 MB of weights, when this stream has its workspace (created on the stream's first
    // such call, never while it is captured); one bf16 vector: the block-diagonal kernel; else
    // the mma.sync kernel (2..8 vectors: 14336 x 4096 Q4_0 at 8 vectors 10.0 against 14.7 us,
    // 151936 x 1024 Q8_0 at 4 vectors 33.8 against 35.6 us; 8 vectors on 175 MB 39.3 against 38.2)
    long long nweights = 0, nbytes = 0;
    for (int i = 0; i < nf; ++i) {
      nweights += fast[i].rows * fast[i].cols;
      nbytes += weight_bytes(fast[i]);
    }
    bool tc = xb && (nb > 8 || (nb >= kTcMinBatch && nbytes >= kTcMinBytes));
    for (int i = 0; i < nf && tc; ++i) tc = decode_tc_supported(fast[i]);
    // float32 activations, 2..8 vectors, launches of 96 MB or more and gated activations: the
    // tensor-memory kernel on the bf16 pairs hi + lo (its 16 MMA columns hold both parts of up
    // to 8 vectors); smaller launches the mma.sync kernel, which splits x in its own stages (one
    // launch: 2048 x 1024 Q4_0 at 8 vectors 3.3 against 7.4 us, 28672 x 4096 at 4 vectors 21.8
    // against 25.7 us; 65536 x 4096 at 8 vectors 61.8 against 50.0 us the other way)
    bool tc32 = !xb && nb >= 2 && (glu || nbytes >= kTcF32MinBytes) && decode_tc_f32_fits(fast, nf);
    for (int i = 0; i < nf && tc32; ++i) tc32 = decode_tc_supported(fast[i]);
    Workspace ws;
    if (tc && stream_workspace(dev, stream, &ws) == cudaSuccess) {
      if (launch_decode_tc(fast, fx, fy, nf, nb, pdl, dev, ws, stream) != cudaSuccess) return QMV_E_CUDA;
    } else if (tc32 && stream_workspace(dev, stream, &ws) == cudaSuccess &&
               launch_decode_tc_f32(fast, fx, fy, nf, nb, pdl, dev, ws, stream, act, batch) ==
                   cudaSuccess) {
      // done (a stream being captured without its split buffer yet falls through to mma.sync)
    } else if (xb && nb == 1) {
      if (launch_matvec_bdiag(fast, fx, fy, nf, pdl, dev, stream) != cudaSuccess) return QMV_E_CUDA;
    } else if (!xb && !glu && nb == 1 && nweights >= kF32SplitMinWeights &&
               nweights * (wtype == QMV_Q8_0 ? 2 : 1) / 2 < kF32InKernelMaxBytes) {
      // one float32 vector: the block-diagonal kernel reads it as float32 and rounds each stage
      // to half after a power-of-two scale, or splits it into bf16 hi + lo parts (one launch;
      // below a few hundred KB of weights the one mma.sync launch measured quicker)
      if (launch_matvec_bdiag_f32in(fast, fx, fy, nf, pdl, dev, stream) != cudaSuccess) return QMV_E_CUDA;
    } else if (!xb && nb == 1 && (glu || nweights >= kF32SplitMinWeights) &&
               launch_matvec_bdiag_f32(fast, fx, fy, nf, pdl, dev, stream, act, batch) == cudaSuccess) {
      // one vector of large launches or of gated activations: x (or act(gate) * up) formed and
      // split into bf16 hi + lo by the split kernel (once per column, not once per row tile),
      // then the block-diagonal kernel on the parts
    } else if (glu) {
      return QMV_E_ARG;  // gated activations need the stream's split buffer (see qmv.h)
    } else if (launch_matvec_mma(fast, fx, fy, nf, xb, nb, pdl, dev, stream) != cudaSuccess) {
      return QMV_E_CUDA;
    }
  }
  return QMV_OK;
}

int qmv_matvec_grouped_noalloc(int wtype, int scale_dtype, int x_dtype, int batch, const qmv_problem* problems,
                               int n, unsigned flags, cudaStream_t stream) {
  if (problems == nullptr || n < 1 || n > QMV_MAX_GROUP) return QMV_E_ARG;
  if (x_dtype != QMV_X_BF16) return QMV_E_FORMAT;  // the tensor-memory kernel reads bf16 only
  if (batch < 0 || batch > QMV_NOALLOC_MAX_BATCH) return QMV_E_ARG;
  if ((flags & ~QMV_FLAG_OVERLAP) != 0) return QMV_E_ARG;
  MatrixRef ms[QMV_MAX_GROUP];
  const void* xs[QMV_MAX_GROUP];
  float* ys[QMV_MAX_GROUP];
  for (int i = 0; i < n; ++i) {
    const qmv_problem& pr = problems[i];
    const int st = make_ref(wtype, scale_dtype, pr.rows, pr.cols, pr.W, &ms[i]);
    if (st != QMV_OK) return st;
    if (!decode_tc_supported(ms[i])) return QMV_E_SHAPE;
    xs[i] = pr.x;
    ys[i] = pr.y;
    if (batch == 0) continue;
    if (pr.x == nullptr || pr.y == nullptr) return QMV_E_ARG;
    if (!aligned(pr.x, 16) || !aligned(pr.y, 4)) return QMV_E_ALIGN;
  }
  if (batch == 0) return QMV_OK;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  void* base = nullptr;
  if (noalloc_scratch(dev.device, &base) != cudaSuccess) return QMV_E_CUDA;
  Workspace ws;
  workspace_carve(base, sizeof(g_noalloc_scratch), QMV_NOALLOC_MAX_CTAS, &ws);
  const bool pdl = (flags & QMV_FLAG_OVERLAP) != 0;
  return launch_decode_tc(ms, xs, ys, n, batch, pdl, dev, ws, stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
}

int qmv_matvec_glu(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void* W1, const void* W3,
                   const void* x, int x_dtype, int act, void* h, unsigned flags, cudaStream_t stream) {
  MatrixRef w1, w3;
  int st = make_ref(wtype, scale_dtype, rows, cols, W1, &w1);
  if (st != QMV_OK) return st;
  st = make_ref(wtype, scale_dtype, rows, cols, W3, &w3);
  if (st != QMV_OK) return st;
  if (wtype != QMV_Q4_0 || x_dtype != QMV_X_BF16) return QMV_E_FORMAT;
  if (act != QMV_ACT_SILU && act != QMV_ACT_GELU_TANH) return QMV_E_FORMAT;
  if ((flags & ~QMV_FLAG_OVERLAP) != 0) return QMV_E_ARG;
  if (!matvec_bdiag_glu_supported(w1, w3)) return QMV_E_SHAPE;
  if (x == nullptr || h == nullptr) return QMV_E_ARG;
  if (!aligned(x, 16) || !aligned(h, 16)) return QMV_E_ALIGN;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  return launch_matvec_bdiag_glu(w1, w3, x, act, static_cast<uint16_t*>(h), (flags & QMV_FLAG_OVERLAP) != 0, dev,
                                 stream) == cudaSuccess
             ? QMV_OK
             : QMV_E_CUDA;
}

int qmv_matvec(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void* W, const void* x,
               int x_dtype, float* y, int batch, cudaStream_t stream) {
  qmv_problem pr;
  pr.rows = rows;
  pr.cols = cols;
  pr.W = W;
  pr.x = x;
  pr.y = y;
  return qmv_matvec_grouped(wtype, scale_dtype, x_dtype, batch, &pr, 1, 0u, stream);
}

int qmv_dequant(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void* W, float* out,
                cudaStream_t stream) {
  MatrixRef m;
  int st = make_ref(wtype, scale_dtype, rows, cols, W, &m);
  if (st != QMV_OK) return st;
  if (out == nullptr) return QMV_E_ARG;
  if (!aligned(out, 16)) return QMV_E_ALIGN;
  return launch_dequant(m, out, stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
}

int qmv_validate(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void* W, int64_t* first_bad,
                 cudaStream_t stream) {
  MatrixRef m;
  int st = make_ref(wtype, scale_dtype, rows, cols, W, &m);
  if (st != QMV_OK) return st;
  if (first_bad == nullptr) return QMV_E_ARG;
  if (!aligned(first_bad, 8)) return QMV_E_ALIGN;
  return launch_validate(m, first_bad, stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
}

int qmv_quantize(int wtype, int scale_dtype, int64_t rows, int64_t cols, const float* src, void* W,
                 int64_t* first_bad, cudaStream_t stream) {
  Layout L;
  const int st = make_layout(wtype, scale_dtype, rows, cols, &L);
  if (st != QMV_OK) return st;
  if (src == nullptr || W == nullptr || first_bad == nullptr) return QMV_E_ARG;
  if (!aligned(src, 16) || !aligned(W, 16) || !aligned(first_bad, 8)) return QMV_E_ALIGN;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  return launch_quantize(wtype, scale_dtype == QMV_SCALE_F16, rows, cols, src, static_cast<uint8_t*>(W), L.d_off,
                         L.q_bytes, first_bad, dev, stream) == cudaSuccess
             ? QMV_OK
             : QMV_E_CUDA;
}

size_t qmv_gguf_bytes(int wtype, int64_t rows, int64_t cols) {
  Layout L;
  if (make_layout(wtype, QMV_SCALE_F16, rows, cols, &L) != QMV_OK) return 0;
  const int64_t nrec = rows * (cols / 32);
  const int64_t rec = wtype == QMV_Q8_0 ? 34 : 18;
  if (nrec > INT64_MAX / rec) return 0;
  return (size_t)(nrec * rec);
}

int qmv_gguf_to_mlb(int wtype, int64_t rows, int64_t cols, const void* src, void* W, cudaStream_t stream) {
  Layout L;
  const int st = make_layout(wtype, QMV_SCALE_F16, rows, cols, &L);
  if (st != QMV_OK) return st;
  if (qmv_gguf_bytes(wtype, rows, cols) == 0) return QMV_E_SHAPE;
  if (src == nullptr || W == nullptr) return QMV_E_ARG;
  if (!aligned(src, 16) || !aligned(W, 16)) return QMV_E_ALIGN;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  return launch_gguf_to_mlb(wtype, rows, cols, src, static_cast<uint8_t*>(W), L.d_off, L.q_bytes, dev, stream) ==
                 cudaSuccess
             ? QMV_OK
             : QMV_E_CUDA;
}

int qmv_quantize_x(int x_dtype, int64_t batch, int64_t cols, const void* x, void* xq, cudaStream_t stream) {
  if (x_dtype != QMV_X_F32 && x_dtype != QMV_X_BF16) return QMV_E_FORMAT;
  if (batch < 0) return QMV_E_ARG;
  if (cols <= 0 || cols % 32 != 0) return QMV_E_SHAPE;
  if (batch == 0) return QMV_OK;
  Layout L;
  const int st = make_layout(QMV_Q8_0, QMV_SCALE_F32, batch, cols, &L);
  if (st != QMV_OK) return st;
  if (x == nullptr || xq == nullptr) return QMV_E_ARG;
  if (!aligned(x, 16) || !aligned(xq, 16)) return QMV_E_ALIGN;
  return launch_quantize_x(x_dtype == QMV_X_BF16, batch, cols, x, static_cast<uint8_t*>(xq), L.d_off, L.q_bytes,
                           stream) == cudaSuccess
             ? QMV_OK
             : QMV_E_CUDA;
}

int qmv_matvec_qx(int wtype, int scale_dtype, int64_t rows, int64_t cols, const void* W, const void* xq,
                  float* y, int batch, cudaStream_t stream) {
  MatrixRef m;
  int st = make_ref(wtype, scale_dtype, rows, cols, W, &m);
  if (st != QMV_OK) return st;
  if (batch < 0) return QMV_E_ARG;
  if (batch == 0) return QMV_OK;
  Layout LX;
  st = make_layout(QMV_Q8_0, QMV_SCALE_F32, batch, cols, &LX);
  if (st != QMV_OK) return st;
  if (xq == nullptr || y == nullptr) return QMV_E_ARG;
  if (!aligned(xq, 16) || !aligned(y, 4)) return QMV_E_ALIGN;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  const int8_t* xqq = static_cast<const int8_t*>(xq);
  const float* xd = reinterpret_cast<const float*>(static_cast<const uint8_t*>(xq) + LX.d_off);
  // 2 or more vectors, cols a multiple of 256: the block dots on the tensor core (quants and
  // levels as exact halves); else the dp4a kernel
  if (batch >= 2 && matvec_mma_supported(m))
    return launch_matvec_qx_mma(&m, &xqq, &xd, 1, batch, &y, false, dev, stream) == cudaSuccess ? QMV_OK
                                                                                                 : QMV_E_CUDA;
  return launch_matvec_qx(m, xqq, xd, batch, y, dev, stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
}

int qmv_matvec_qx_grouped(int wtype, int scale_dtype, int x_dtype, int batch, const qmv_problem* problems, int n,
                          unsigned flags, cudaStream_t stream) {
  if (problems == nullptr || n < 1 || n > QMV_MAX_GROUP) return QMV_E_ARG;
  if (x_dtype != QMV_X_F32 && x_dtype != QMV_X_BF16) return QMV_E_FORMAT;
  if (batch < 0) return QMV_E_ARG;
  if ((flags & ~QMV_FLAG_OVERLAP) != 0) return QMV_E_ARG;
  MatrixRef ms[QMV_MAX_GROUP];
  const void* xs[QMV_MAX_GROUP];
  float* ys[QMV_MAX_GROUP];
  const int64_t nv = batch < 8 ? batch : 8;
  for (int i = 0; i < n; ++i) {
    const qmv_problem& pr = problems[i];
    const int st = make_ref(wtype, scale_dtype, pr.rows, pr.cols, pr.W, &ms[i]);
    if (st != QMV_OK) return st;
    if (nv * pr.cols > QMV_QX_MAX_VEC_COLS) return QMV_E_SHAPE;
    xs[i] = pr.x;
    ys[i] = pr.y;
    if (batch == 0) continue;
    if (pr.x == nullptr || pr.y == nullptr) return QMV_E_ARG;
    if (!aligned(pr.x, 16) || !aligned(pr.y, 4)) return QMV_E_ALIGN;
    if (pr.rows > INT64_MAX / batch) return QMV_E_SHAPE;
  }
  if (batch == 0) return QMV_OK;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  // one vector, every problem's cols a multiple of 256, under 96 MB of weights: the
  // block-diagonal kernel quantizes the activations in its stages and takes the block dots on
  // the tensor core (exact integer sums in half precision); else the fused dp4a kernel (whose
  // quantizing prologue is paid once per CTA: on a 151 MB launch it measured 28.4 against
  // 31.7 us, on the layer's launches of 9.4 to 51 MB 3 to 30% slower)
  bool bdiag = batch == 1;
  long long qx_bytes = 0;
  for (int i = 0; i < n && bdiag; ++i) {
    bdiag = matvec_mma_supported(ms[i]);
    qx_bytes += ms[i].rows * ms[i].cols / 32 * ((wtype == QMV_Q4_0 ? 16 : 32) + (scale_dtype == QMV_SCALE_F16 ? 2 : 4));
  }
  if (qx_bytes >= kQxBdiagMaxBytes) bdiag = false;
  if (bdiag)
    return launch_matvec_bdiag_qx(ms, xs, ys, n, x_dtype == QMV_X_BF16, (flags & QMV_FLAG_OVERLAP) != 0, dev,
                                  stream) == cudaSuccess
               ? QMV_OK
               : QMV_E_CUDA;
  // two or more vectors, every problem's cols a multiple of 256, the images within the stream's
  // split buffer: a quantizer launch writes each distinct activation array's image there (the
  // bytes qmv_quantize_x writes), then the tensor-core mode of the mma.sync kernel, launched as
  // its programmatic dependent, takes the block dots (65536 x 4096 Q4_0 at 8 vectors: about half
  // the dp4a kernel's time, whose CTAs each quantize the activations again)
  bool two_step = batch >= 2;
  for (int i = 0; i < n && two_step; ++i) two_step = matvec_mma_supported(ms[i]);
  if (two_step) {
    QxImages im{};
    int owner[QMV_MAX_GROUP];  // the image problem i reads
    int nim = 0;
    size_t need = 0;
    auto round256 = [](size_t b) { return (b + 255) / 256 * 256; };
    for (int i = 0; i < n; ++i) {
      owner[i] = -1;
      for (int j = 0; j < i && owner[i] < 0; ++j)
        if (xs[j] == xs[i] && ms[j].cols == ms[i].cols) owner[i] = owner[j];
      if (owner[i] >= 0) continue;
      owner[i] = nim;
      im.x[nim] = xs[i];
      im.nblk[nim] = (long long)batch * (ms[i].cols / 32);
      need += round256((size_t)batch * (size_t)ms[i].cols) + round256((size_t)im.nblk[nim] * 4);
      ++nim;
    }
    // (a stream captured before its first such call has no buffer yet: the dp4a kernel then)
    uint8_t* base = nullptr;
    two_step = need <= split_buffer_bytes() && stream_split_buffer(dev, stream, &base) == cudaSuccess;
    if (two_step) {
      for (int k = 0; k < nim; ++k) {
        im.q[k] = base;
        base += round256((size_t)im.nblk[k] * 32);
        im.d[k] = reinterpret_cast<float*>(base);
        base += round256((size_t)im.nblk[k] * 4);
      }
      if (launch_quantize_x_group(x_dtype == QMV_X_BF16, im, nim, (flags & QMV_FLAG_OVERLAP) != 0, stream) !=
          cudaSuccess)
        return QMV_E_CUDA;
      const int8_t* xq[QMV_MAX_GROUP];
      const float* xd[QMV_MAX_GROUP];
      for (int i = 0; i < n; ++i) {
        xq[i] = reinterpret_cast<const int8_t*>(im.q[owner[i]]);
        xd[i] = im.d[owner[i]];
      }
      return launch_matvec_qx_mma(ms, xq, xd, n, batch, ys, true, dev, stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
    }
  }
  return launch_matvec_qx_fused(ms, xs, ys, n, x_dtype == QMV_X_BF16, batch, (flags & QMV_FLAG_OVERLAP) != 0, dev,
                                stream) == cudaSuccess
             ? QMV_OK
             : QMV_E_CUDA;
}

int qmv_quantize_q4_fit(int scale_dtype, int64_t rows, int64_t cols, const float* src, void* W, int64_t* first_bad,
                        cudaStream_t stream) {
  Layout L;
  const int st = make_layout(QMV_Q4_0, scale_dtype, rows, cols, &L);
  if (st != QMV_OK) return st;
  if (src == nullptr || W == nullptr || first_bad == nullptr) return QMV_E_ARG;
  if (!aligned(src, 16) || !aligned(W, 16) || !aligned(first_bad, 8)) return QMV_E_ALIGN;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  return launch_quantize(kQuantQ4Fit, scale_dtype == QMV_SCALE_F16, rows, cols, src, static_cast<uint8_t*>(W), L.d_off,
                         L.q_bytes, first_bad, dev, stream) == cudaSuccess
             ? QMV_OK
             : QMV_E_CUDA;
}

int qmv_check_device(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return QMV_E_CUDA;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return QMV_E_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return QMV_E_CUDA;
    // a kernel that gave up may have left a split tile's arrival counter part-way
    if (reset_workspaces() != cudaSuccess) return QMV_E_CUDA;
    if (noalloc_reset(dev.device) != cudaSuccess) return QMV_E_CUDA;
  }
  return v;
}

const char* qmv_strerror(int status) {
  switch (status) {
    case QMV_OK: return "ok";
    case QMV_E_FORMAT: return "format error (unknown wtype/scale/x dtype, or an invalid quant)";
    case QMV_E_SHAPE: return "shape error (zero dimension, cols not a multiple of 32, or size overflow)";
    case QMV_E_ARG: return "invalid argument (null pointer or negative batch)";
    case QMV_E_ALIGN: return "misaligned pointer (W and x need 16 bytes, y 4, out 16, first_bad 8)";
    case QMV_E_CUDA: return "CUDA error (launch failed, no device, or no sm_103a device)";
    case QMV_E_TIMEOUT: return "a kernel's bounded wait ran out; its output is incomplete";
    default: return "unknown status";
  }
}

}  // extern "C"
