// step.cu -- compiled steps: a fixed sequence of copies and grouped products, run once eagerly
// on a private stream (which sets up the kernels and that stream's workspaces and checks the
// arguments), then recorded as a CUDA graph and replayed by one call per step.  The graph's
// kernels hold the private stream's workspace pointers, so a step owns its workspaces and two
// steps never share them.
#include <new>

#include "qmv.h"
#include "qmv_common.cuh"
#include "qmv_internal.h"

struct qmv_step {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  cudaStream_t cap;  // the private stream the step was recorded on (keys its workspaces)
  int device;
};

namespace {

// A copy between device memory and pinned host memory done by the GPU's own loads and stores
// through the host memory's device address (a kernel node in the step's graph costs less than
// a copy node for the few KB a decode step moves).  16-byte pieces when both ends and the size
// allow it, bytes otherwise.  The products that follow may start (programmatic launch); they
// wait for this kernel before reading what it wrote.
__global__ void __launch_bounds__(256) step_copy_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                        size_t bytes) {
  if (threadIdx.x == 0) qmv::griddep_launch_dependents();
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | bytes) & 15u) == 0) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (size_t i = tid; i < bytes / 16; i += stride) d[i] = s[i];
  } else {
    for (size_t i = tid; i < bytes; i += stride) dst[i] = src[i];
  }
}

// The device address of pinned host memory at p (mapped into the device's address space), or
// null when p is not such memory.
void* host_device_address(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // a pointer the runtime does not know: clear the error
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost) return nullptr;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  // with unified addressing the device address is the host address; anything else takes the
  // runtime's copy
  return d == p ? d : nullptr;
}

bool is_device(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice;
}

// One copy of the step: a kernel between device memory and mapped pinned host memory, else
// cudaMemcpyAsync.
cudaError_t copy(const qmv_copy& c, cudaStream_t s) {
  if (c.bytes == 0) return cudaSuccess;
  const void* src = c.src;
  void* dst = c.dst;
  void* hs = host_device_address(c.src);
  void* hd = host_device_address(c.dst);
  if (hs != nullptr && hd == nullptr && is_device(c.dst)) src = hs;
  else if (hd != nullptr && hs == nullptr && is_device(c.src)) dst = hd;
  else return cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDefault, s);
  const size_t pieces = (c.bytes + 15) / 16;
  unsigned grid = (unsigned)((pieces + 255) / 256);
  if (grid > 64) grid = 64;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, step_copy_kernel, static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
                            c.bytes);
}

// The step's sequence on `s`: the first failing call's status.
int enqueue(const qmv_copy* before, int n_before, const qmv_group* groups, int n_groups, const qmv_copy* after,
            int n_after, cudaStream_t s) {
  for (int i = 0; i < n_before; ++i)
    if (copy(before[i], s) != cudaSuccess) return QMV_E_CUDA;
  for (int i = 0; i < n_groups; ++i) {
    const qmv_group& g = groups[i];
    const int st = qmv_matvec_grouped(g.wtype, g.scale_dtype, g.x_dtype, g.batch, g.problems, g.n, g.flags, s);
    if (st != QMV_OK) return st;
  }
  for (int i = 0; i < n_after; ++i)
    if (copy(after[i], s) != cudaSuccess) return QMV_E_CUDA;
  return QMV_OK;
}

bool copies_ok(const qmv_copy* c, int n) {
  if (n < 0 || (n > 0 && c == nullptr)) return false;
  for (int i = 0; i < n; ++i)
    if (c[i].bytes > 0 && (c[i].dst == nullptr || c[i].src == nullptr)) return false;
  return true;
}

void discard(cudaStream_t cap, int device) {
  cudaStreamSynchronize(cap);
  qmv::release_stream_workspaces(device, cap);
  cudaStreamDestroy(cap);
}

}  // namespace

extern "C" {

int qmv_step_create(const qmv_copy* before, int n_before, const qmv_group* groups, int n_groups,
                    const qmv_copy* after, int n_after, qmv_step** step) {
  if (step == nullptr) return QMV_E_ARG;
  *step = nullptr;
  if (!copies_ok(before, n_before) || !copies_ok(after, n_after)) return QMV_E_ARG;
  if (n_groups < 0 || (n_groups > 0 && groups == nullptr)) return QMV_E_ARG;
  qmv::DeviceInfo dev;
  if (qmv::current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  cudaStream_t cap = nullptr;
  if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) return QMV_E_CUDA;
  if (qmv::prepare_stream_workspaces(dev, cap) != cudaSuccess) {
    discard(cap, dev.device);
    return QMV_E_CUDA;
  }
  // the eager run: kernel attributes, checks of every argument
  int st = enqueue(before, n_before, groups, n_groups, after, n_after, cap);
  if (st == QMV_OK && cudaStreamSynchronize(cap) != cudaSuccess) st = QMV_E_CUDA;
  if (st != QMV_OK) {
    discard(cap, dev.device);
    return st;
  }
  // the recording
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    discard(cap, dev.device);
    return QMV_E_CUDA;
  }
  st = enqueue(before, n_before, groups, n_groups, after, n_after, cap);
  cudaGraph_t graph = nullptr;
  const cudaError_t end = cudaStreamEndCapture(cap, &graph);  // always ends the capture
  cudaGraphExec_t exec = nullptr;
  if (st == QMV_OK && (end != cudaSuccess || graph == nullptr)) st = QMV_E_CUDA;
  if (st == QMV_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) st = QMV_E_CUDA;
  qmv_step* s = nullptr;
  if (st == QMV_OK) {
    s = new (std::nothrow) qmv_step{graph, exec, cap, dev.device};
    if (s == nullptr) st = QMV_E_CUDA;
  }
  if (st != QMV_OK) {
    if (exec != nullptr) cudaGraphExecDestroy(exec);
    if (graph != nullptr) cudaGraphDestroy(graph);
    discard(cap, dev.device);
    return st;
  }
  *step = s;
  return QMV_OK;
}

int qmv_step_run(qmv_step* step, cudaStream_t stream) {
  if (step == nullptr) return QMV_E_ARG;
  return cudaGraphLaunch(step->exec, stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
}

int qmv_step_run_wait(qmv_step* step, cudaStream_t stream) {
  if (step == nullptr) return QMV_E_ARG;
  if (cudaGraphLaunch(step->exec, stream) != cudaSuccess) return QMV_E_CUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
}

int qmv_step_destroy(qmv_step* step) {
  if (step == nullptr) return QMV_OK;
  int st = cudaDeviceSynchronize() == cudaSuccess ? QMV_OK : QMV_E_CUDA;
  if (cudaGraphExecDestroy(step->exec) != cudaSuccess) st = QMV_E_CUDA;
  if (cudaGraphDestroy(step->graph) != cudaSuccess) st = QMV_E_CUDA;
  if (qmv::release_stream_workspaces(step->device, step->cap) != cudaSuccess) st = QMV_E_CUDA;
  if (cudaStreamDestroy(step->cap) != cudaSuccess) st = QMV_E_CUDA;
  delete step;
  return st;
}

}  // extern "C"
