// step.cu -- compiled steps: a fixed sequence of copies and grouped products, run once eagerly
// on a private stream (which sets up the kernels and that stream's workspaces and checks the
// arguments), then recorded as a CUDA graph and replayed by one call per step.  The graph's
// kernels hold the private stream's workspace pointers, so a step owns its workspaces and two
// steps never share them.
#include <new>

#include "qmv.h"
#include "qmv_internal.h"

struct qmv_step {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  cudaStream_t cap;  // the private stream the step was recorded on (keys its workspaces)
  int device;
};

namespace {

// The step's sequence on `s`: the first failing call's status.
int enqueue(const qmv_copy* before, int n_before, const qmv_group* groups, int n_groups, const qmv_copy* after,
            int n_after, cudaStream_t s) {
  for (int i = 0; i < n_before; ++i)
    if (cudaMemcpyAsync(before[i].dst, before[i].src, before[i].bytes, cudaMemcpyDefault, s) != cudaSuccess)
      return QMV_E_CUDA;
  for (int i = 0; i < n_groups; ++i) {
    const qmv_group& g = groups[i];
    const int st = qmv_matvec_grouped(g.wtype, g.scale_dtype, g.x_dtype, g.batch, g.problems, g.n, g.flags, s);
    if (st != QMV_OK) return st;
  }
  for (int i = 0; i < n_after; ++i)
    if (cudaMemcpyAsync(after[i].dst, after[i].src, after[i].bytes, cudaMemcpyDefault, s) != cudaSuccess)
      return QMV_E_CUDA;
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
