// decode_tc.cu -- entry of the tensor-memory decode product (kernels in decode_tc.cuh) and
// the per-stream workspace its split tiles use.
#include <map>
#include <mutex>
#include <utility>

#include "decode_tc.cuh"

namespace qmv {

bool decode_tc_supported(const MatrixRef& m) {
  return m.cols % dtc::kKS == 0 && m.rows < (1LL << 31) - dtc::kTileRows && m.cols < (1LL << 30);
}

int decode_tc_max_problems() { return dtc::kMaxProblems; }

size_t workspace_counter_bytes(int n) { return ((size_t)n * sizeof(unsigned) + 255) / 256 * 256; }

void workspace_carve(void* base, size_t bytes, int n, Workspace* ws) {
  const size_t cb = workspace_counter_bytes(n);
  ws->counters = static_cast<unsigned*>(base);
  ws->max_counters = n;
  ws->partials = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + cb);
  ws->max_partial_floats = bytes > cb ? (bytes - cb) / sizeof(float) : 0;
}

// a stream's workspace: counters for up to 1024 CTAs, then the parts (2 per CTA of 128
// rows x up to 16 vectors); the kernel sizes its grid to fit
constexpr int kStreamCounters = 1024;
constexpr size_t kStreamWorkspaceBytes = (size_t)8 << 20;

// a stream's prefill workspace: counters for 4096 tiles, then the parts of split tiles
// (ksplit x 128 rows x up to 128 vectors per tile; the launch picks ksplit to fit)
constexpr int kPrefillCounters = 4096;
constexpr size_t kPrefillWorkspaceBytes = (size_t)32 << 20;

// a stream's buffer for float32 activations split into bfloat16 pairs (16 rows of cols
// bf16 per problem: up to 65,536 columns over the problems of one launch)
constexpr size_t kSplitBytes = (size_t)2 << 20;

namespace {
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
std::map<std::pair<int, cudaStream_t>, Workspace> g_pws;
std::map<std::pair<int, cudaStream_t>, Workspace> g_xws;

cudaError_t cached_workspace(std::map<std::pair<int, cudaStream_t>, Workspace>& cache, const DeviceInfo& dev,
                             cudaStream_t stream, size_t bytes, int counters, Workspace* ws) {
  constexpr size_t kMaxEntries = 64;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  const auto key = std::make_pair(dev.device, stream);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *ws = it->second;
    return cudaSuccess;
  }
  if (cache.size() >= kMaxEntries) return cudaErrorMemoryAllocation;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t err = cudaStreamIsCapturing(stream, &cs);
  if (err != cudaSuccess) return err;
  if (cs != cudaStreamCaptureStatusNone) return cudaErrorNotReady;  // no allocation while capturing
  void* base = nullptr;
  err = cudaMalloc(&base, bytes);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(base, 0, workspace_counter_bytes(counters), stream);
  if (err != cudaSuccess) {
    cudaFree(base);
    return err;
  }
  Workspace w;
  workspace_carve(base, bytes, counters, &w);
  cache.emplace(key, w);
  *ws = w;
  return cudaSuccess;
}
}  // namespace

cudaError_t stream_workspace(const DeviceInfo& dev, cudaStream_t stream, Workspace* ws) {
  return cached_workspace(g_ws, dev, stream, kStreamWorkspaceBytes, kStreamCounters, ws);
}

cudaError_t stream_prefill_workspace(const DeviceInfo& dev, cudaStream_t stream, Workspace* ws) {
  return cached_workspace(g_pws, dev, stream, kPrefillWorkspaceBytes, kPrefillCounters, ws);
}

namespace {

struct SplitArgs {
  const float* x[dtc::kMaxProblems];
  uint16_t* out[dtc::kMaxProblems];
  int cols[dtc::kMaxProblems];
  int batch;
  int nvec;    // hi rows written (the lo rows too): batch rounded up to the consumer's width
  int lo_row;  // row of vector 0's lo part
  int act;     // -1: x as given; 0 / 1: x is a gate and the activations are act(gate) * up
  long long up_batch;  // gated activations: a problem's up array is up_batch * cols floats after its gate
};

// x (batch float32 vectors of cols) as rows of bfloat16: row n < nvec the hi part of vector
// n, row lo_row + n its lo part, hi = RN_bf16(x) and lo = RN_bf16(x - hi) (x - hi is exact
// in float32); rows of vectors past the batch are zero, and so is lo of a value that is not
// finite.  One thread per column of one problem (blockIdx.y).
__global__ void __launch_bounds__(256) split_x_kernel(const __grid_constant__ SplitArgs a) {
  griddep_wait();  // the activations may be the preceding kernel's output
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int i = blockIdx.y;
  const int cols = a.cols[i];
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  const float* x = a.x[i];
  uint16_t* out = a.out[i];
  for (int n = 0; n < a.nvec; ++n) {
    uint16_t hi = 0, lo = 0;
    if (n < a.batch) {
      float v = x[(size_t)n * cols + c];
      if (a.act >= 0) v = glu(a.act, v, x[(size_t)(a.up_batch + n) * cols + c]);
      split_bf16_pair(v, hi, lo);
    }
    out[(size_t)n * cols + c] = hi;
    out[(size_t)(a.lo_row + n) * cols + c] = lo;
  }
}

// The block-diagonal kernel's half route for one float32 vector per problem (or act(gate) * up):
// per column the bfloat16 pair hi, lo (rows 0 and 1, split_x_kernel's rule) and, per 256-column
// chunk, the power of two xs = 2^s that brings the chunk's largest magnitude into [2^14, 2^15)
// (half_stage_scale): row 2 holds RN_half(x * xs) and, after the three rows, one float per chunk
// holds 2^-s, or 0 when the chunk does not round (a value not finite, or a nonzero value with
// |x * xs| under 2^-14, where half is not normal), whose products take hi and lo instead.  One
// CTA of 256 threads per chunk (blockIdx.x) of a problem (blockIdx.y).
struct HalfSplitArgs {
  const float* x[dtc::kMaxProblems];
  uint16_t* out[dtc::kMaxProblems];
  int cols[dtc::kMaxProblems];
  int act;             // -1: x as given; 0 / 1: x is a gate and the activations are act(gate) * up
  long long up_batch;  // gated activations: a problem's up array is up_batch * cols floats after its gate
};

__global__ void __launch_bounds__(256) split_x_half_kernel(const __grid_constant__ HalfSplitArgs a) {
  griddep_wait();  // the activations may be the preceding kernel's output
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int i = blockIdx.y;
  const int cols = a.cols[i];
  if ((int)blockIdx.x * 256 >= cols) return;  // the whole CTA: past this problem's chunks
  const int c = blockIdx.x * 256 + threadIdx.x;
  const float* x = a.x[i];
  float v = x[c];
  if (a.act >= 0) v = glu(a.act, v, x[(size_t)a.up_batch * cols + c]);
  uint16_t hi, lo;
  split_bf16_pair(v, hi, lo);
  uint16_t* out = a.out[i];
  out[c] = hi;
  out[cols + c] = lo;
  // the chunk's largest magnitude and smallest nonzero magnitude, as float32 bit patterns
  // (unsigned order is magnitude order; a NaN lies above infinity)
  const uint32_t m = __float_as_uint(v) & 0x7FFFFFFFu;
  __shared__ uint32_t wmax[8], wmin[8];
  uint32_t amax = __reduce_max_sync(0xffffffffu, m);
  uint32_t amin = __reduce_min_sync(0xffffffffu, m == 0u ? 0xFFFFFFFFu : m);
  if ((threadIdx.x & 31) == 0) {
    wmax[threadIdx.x >> 5] = amax;
    wmin[threadIdx.x >> 5] = amin;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    amax = wmax[w] > amax ? wmax[w] : amax;
    amin = wmin[w] < amin ? wmin[w] : amin;
  }
  float xs, xinv;
  bool fits = amax <= 0x7F7FFFFFu && half_stage_scale(__uint_as_float(amax), xs, xinv);
  if (fits && amin != 0xFFFFFFFFu) fits = __uint_as_float(amin) * xs >= 0x1p-14f;
  out[2 * cols + c] = __half_as_ushort(__float2half_rn(fits ? v * xs : 0.f));
  if (threadIdx.x == 0) reinterpret_cast<float*>(out + 3 * (size_t)cols)[blockIdx.x] = fits ? xinv : 0.f;
}

// Bytes of one problem's area of the half route's buffer (three rows of cols two-byte values and
// cols / 256 floats), rounded up to 512 so that every row of the next problem stays aligned.
size_t half_area_bytes(int64_t cols) { return ((size_t)cols * 6 + (size_t)cols / 64 + 511) / 512 * 512; }

}  // namespace

// Split the float32 activations of n problems (batch vectors each) into rows of bfloat16 in
// the stream's split buffer: per problem lo_row + nvec rows of cols, laid out one problem
// after the other; sx[i] receives problem i's rows.  pdl: the split waits for the preceding
// kernel before reading x.
static cudaError_t split_activations(const MatrixRef* ms, const void* const* xs, int n, int batch, int nvec, int lo_row,
                                     int act, long long up_batch, bool pdl, const DeviceInfo& dev, cudaStream_t stream,
                                     const void** sx) {
  if (n < 1 || n > dtc::kMaxProblems || batch < 1 || batch > nvec) return cudaErrorInvalidValue;
  const int rows = lo_row + nvec;
  size_t need = 0;
  int maxcols = 0;
  for (int i = 0; i < n; ++i) {
    need += (size_t)rows * (size_t)ms[i].cols * 2;
    if (ms[i].cols > maxcols) maxcols = (int)ms[i].cols;
  }
  if (need > kSplitBytes) return cudaErrorInvalidValue;
  Workspace xw;
  cudaError_t err = cached_workspace(g_xws, dev, stream, kSplitBytes, 0, &xw);
  if (err != cudaSuccess) return err;
  SplitArgs a{};
  uint8_t* base = reinterpret_cast<uint8_t*>(xw.partials);
  for (int i = 0; i < n; ++i) {
    a.x[i] = static_cast<const float*>(xs[i]);
    a.out[i] = reinterpret_cast<uint16_t*>(base);
    a.cols[i] = (int)ms[i].cols;
    sx[i] = base;
    base += (size_t)rows * (size_t)ms[i].cols * 2;  // cols % 256 == 0: every row 512-byte aligned
  }
  a.batch = batch;
  a.nvec = nvec;
  a.lo_row = lo_row;
  a.act = act;
  a.up_batch = up_batch;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((maxcols + 255) / 256), (unsigned)n);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, split_x_kernel, a);
}

cudaError_t launch_decode_tc_f32(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch,
                                 bool pdl, const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream, int act,
                                 long long up_batch) {
  const void* sx[dtc::kMaxProblems];
  // 16 MMA columns: the hi parts of up to 8 vectors, then their lo parts
  cudaError_t err =
      split_activations(ms, xs, n, batch, dtc::kMaxBatch, dtc::kMaxBatch, act, up_batch, pdl, dev, stream, sx);
  if (err != cudaSuccess) return err;
  // the product launches as a programmatic dependent of the split: its weight loads overlap it
  if (ms[0].wtype == QMV_Q4_0) return dtc::launch_q4(ms, sx, ys, n, batch, true, true, dev, ws, stream);
  return dtc::launch_q8(ms, sx, ys, n, batch, true, true, dev, ws, stream);
}

bool decode_tc_f32_fits(const MatrixRef* ms, int n) {
  size_t need = 0;
  for (int i = 0; i < n; ++i) need += (size_t)dtc::kN * (size_t)ms[i].cols * 2;
  return need <= kSplitBytes;
}

cudaError_t launch_matvec_bdiag_f32(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, bool pdl,
                                    const DeviceInfo& dev, cudaStream_t stream, int act, long long up_batch) {
  if (n < 1 || n > dtc::kMaxProblems) return cudaErrorInvalidValue;
  size_t need = 0;
  int maxcols = 0;
  for (int i = 0; i < n; ++i) {
    if (ms[i].cols % dtc::kKS != 0) return cudaErrorInvalidValue;
    need += half_area_bytes(ms[i].cols);
    if (ms[i].cols > maxcols) maxcols = (int)ms[i].cols;
  }
  if (need > kSplitBytes) return cudaErrorInvalidValue;
  Workspace xw;
  cudaError_t err = cached_workspace(g_xws, dev, stream, kSplitBytes, 0, &xw);
  if (err != cudaSuccess) return err;
  HalfSplitArgs a{};
  const void* sx[dtc::kMaxProblems];
  uint8_t* base = reinterpret_cast<uint8_t*>(xw.partials);
  for (int i = 0; i < n; ++i) {
    a.x[i] = static_cast<const float*>(xs[i]);
    a.out[i] = reinterpret_cast<uint16_t*>(base);
    a.cols[i] = (int)ms[i].cols;
    sx[i] = base;
    base += half_area_bytes(ms[i].cols);
  }
  a.act = act;
  a.up_batch = up_batch;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(maxcols / dtc::kKS), (unsigned)n);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  err = cudaLaunchKernelEx(&cfg, split_x_half_kernel, a);
  if (err != cudaSuccess) return err;
  // the product launches as a programmatic dependent of the split: its weight loads overlap it
  return launch_matvec_bdiag_half(ms, sx, ys, n, true, dev, stream);
}

cudaError_t reset_workspaces() {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  for (auto* cache : {&g_ws, &g_pws}) {
    for (auto& kv : *cache) {
      if (kv.first.first != dev) continue;
      err = cudaMemset(kv.second.counters, 0, workspace_counter_bytes(kv.second.max_counters));
      if (err != cudaSuccess) return err;
    }
  }
  return cudaDeviceSynchronize();
}

size_t split_buffer_bytes() { return kSplitBytes; }

cudaError_t stream_split_buffer(const DeviceInfo& dev, cudaStream_t stream, uint8_t** base) {
  Workspace xw;
  const cudaError_t err = cached_workspace(g_xws, dev, stream, kSplitBytes, 0, &xw);
  if (err != cudaSuccess) return err;
  *base = reinterpret_cast<uint8_t*>(xw.partials);
  return cudaSuccess;
}

cudaError_t prepare_stream_workspaces(const DeviceInfo& dev, cudaStream_t stream) {
  Workspace w;
  cudaError_t err = cached_workspace(g_ws, dev, stream, kStreamWorkspaceBytes, kStreamCounters, &w);
  if (err != cudaSuccess) return err;
  err = cached_workspace(g_pws, dev, stream, kPrefillWorkspaceBytes, kPrefillCounters, &w);
  if (err != cudaSuccess) return err;
  return cached_workspace(g_xws, dev, stream, kSplitBytes, 0, &w);
}

cudaError_t release_stream_workspaces(int device, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  cudaError_t first = cudaSuccess;
  for (auto* cache : {&g_ws, &g_pws, &g_xws}) {
    auto it = cache->find(std::make_pair(device, stream));
    if (it == cache->end()) continue;
    const cudaError_t err = cudaFree(it->second.counters);  // the allocation's base
    if (err != cudaSuccess && first == cudaSuccess) first = err;
    cache->erase(it);
  }
  return first;
}

cudaError_t launch_decode_tc(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch, bool pdl,
                             const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream) {
  if (ms[0].wtype == QMV_Q4_0) return dtc::launch_q4(ms, xs, ys, n, batch, false, pdl, dev, ws, stream);
  return dtc::launch_q8(ms, xs, ys, n, batch, false, pdl, dev, ws, stream);
}

}  // namespace qmv
