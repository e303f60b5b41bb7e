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

// a stream's workspace: counters for up to 1024 CTAs, then the parts (2 per CTA of 256
// rows x 8 vectors); the kernel sizes its grid to fit
constexpr int kStreamCounters = 1024;
constexpr size_t kStreamWorkspaceBytes = (size_t)4 << 20;

// a stream's prefill workspace: counters for 4096 tiles, then the parts of split tiles
// (ksplit x 128 rows x up to 128 vectors per tile; the launch picks ksplit to fit)
constexpr int kPrefillCounters = 4096;
constexpr size_t kPrefillWorkspaceBytes = (size_t)32 << 20;

namespace {
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
std::map<std::pair<int, cudaStream_t>, Workspace> g_pws;

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

cudaError_t launch_decode_tc(const MatrixRef* ms, const void* const* xs, float* const* ys, int n, int batch, bool pdl,
                             const DeviceInfo& dev, const Workspace& ws, cudaStream_t stream) {
  if (ms[0].wtype == QMV_Q4_0) return dtc::launch_q4(ms, xs, ys, n, batch, pdl, dev, ws, stream);
  return dtc::launch_q8(ms, xs, ys, n, batch, pdl, dev, ws, stream);
}

}  // namespace qmv
