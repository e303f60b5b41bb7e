// step.cu -- compiled steps: a fixed sequence of copies and grouped products, run once eagerly
// on a private stream (which sets up the kernels and that stream's workspaces and checks the
// arguments), then recorded as a CUDA graph and replayed by one call per step.  The graph's
// kernels hold the private stream's workspace pointers, so a step owns its workspaces and two
// steps never share them.  A gated step's graph starts with a kernel that waits until the host
// opens the run (a count in pinned host memory) and then copies the step's inputs from pinned
// host memory, and ends with a kernel that reports the run done the same way: a decode loop
// enqueues the next token's run while the current one computes and only opens it later.
#include <chrono>
#include <new>

#include "qmv.h"
#include "qmv_common.cuh"
#include "qmv_internal.h"

struct qmv_step {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  cudaStream_t cap;  // the private stream the step was recorded on (keys its workspaces)
  int device;
  // a gated step: the run's first kernel waits until the host opens it (flags[0]), and its last
  // kernel reports the run done (flags[1]); both words are pinned host memory the device
  // addresses directly, the run counter the kernels keep (dev_seq) device memory
  bool gated;
  unsigned long long* flags;
  unsigned long long* dev_seq;
  unsigned long long submitted, opened;  // runs enqueued and opened by the host
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

// A gated run's first kernel: every CTA waits (thread 0 polling, a bound of one second on the
// global timer) until the host's open count reaches this run's number (the runs the step's last
// kernel has counted, plus one), then all CTAs copy the step's `before` copies (mapped pinned
// host memory to device memory) in 16-byte pieces where both ends and the size allow, bytes
// otherwise.  The step's products may launch at once (programmatic dependents) and load their
// first weights while the run waits for the host; they read what this kernel writes only after
// it has finished.
constexpr int kGateCopies = 8;
struct GateCopies {
  const uint8_t* src[kGateCopies];
  uint8_t* dst[kGateCopies];
  size_t bytes[kGateCopies];
  int n;
};

__device__ __forceinline__ unsigned long long ld_acquire_sys(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(256) step_gate_kernel(const unsigned long long* __restrict__ open_count,
                                                        const unsigned long long* __restrict__ dev_seq,
                                                        const __grid_constant__ GateCopies c, int* status) {
  if (threadIdx.x == 0) qmv::griddep_launch_dependents();
  if (threadIdx.x == 0) {
    const unsigned long long want = *dev_seq + 1;
    const unsigned long long t0 = global_ns();
    while (ld_acquire_sys(open_count) < want) {
      if (global_ns() - t0 > 1000000000ull) {  // the host never opened the run
        qmv::record_status(status, QMV_E_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
  }
  __syncthreads();
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (int k = 0; k < c.n; ++k) {
    const uint8_t* src = c.src[k];
    uint8_t* dst = c.dst[k];
    const size_t bytes = c.bytes[k];
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | bytes) & 15u) == 0) {
      const uint4* s = reinterpret_cast<const uint4*>(src);
      uint4* d = reinterpret_cast<uint4*>(dst);
      for (size_t i = tid; i < bytes / 16; i += stride) d[i] = s[i];
    } else {
      for (size_t i = tid; i < bytes; i += stride) dst[i] = src[i];
    }
  }
}

// A gated run's last kernel (one thread, after everything else of the run): counts the run and
// publishes the count to the host after a system-wide fence, so that the host, having read the
// count, also sees every result the run stored into host memory.  Launched as a programmatic
// dependent of the run's last kernel (resident before that kernel ends); it waits for it first.
__global__ void step_done_kernel(unsigned long long* done_count, unsigned long long* dev_seq) {
  qmv::griddep_wait();
  const unsigned long long seq = *dev_seq + 1;
  *dev_seq = seq;
  __threadfence_system();
  asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(done_count), "l"(seq) : "memory");
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

// The gate of a gated step: its `before` copies, each between mapped pinned host memory and
// device memory (the gate kernel performs them), at most kGateCopies.
bool gate_copies(const qmv_copy* before, int n_before, GateCopies* g) {
  if (n_before > kGateCopies) return false;
  *g = GateCopies{};
  for (int i = 0; i < n_before; ++i) {
    void* hs = host_device_address(before[i].src);
    if (before[i].bytes > 0 && (hs == nullptr || !is_device(before[i].dst))) return false;
    g->src[g->n] = static_cast<const uint8_t*>(hs);
    g->dst[g->n] = static_cast<uint8_t*>(before[i].dst);
    g->bytes[g->n] = before[i].bytes;
    ++g->n;
  }
  return true;
}

// The step's sequence on `s`: the first failing call's status.  gate: the gated step's flags
// and counter (its `before` copies are then the gate kernel's), else null.
int enqueue(const qmv_copy* before, int n_before, const qmv_group* groups, int n_groups, const qmv_copy* after,
            int n_after, cudaStream_t s, const qmv_step* gate = nullptr) {
  if (gate != nullptr) {
    GateCopies g;
    if (!gate_copies(before, n_before, &g)) return QMV_E_ARG;
    size_t most = 16;
    for (int k = 0; k < g.n; ++k) most = g.bytes[k] > most ? g.bytes[k] : most;
    const size_t pieces = (most + 15) / 16;
    unsigned grid = (unsigned)((pieces + 255) / 256);
    if (grid > 64) grid = 64;
    qmv::DeviceInfo dev;
    if (qmv::current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
    step_gate_kernel<<<grid, 256, 0, s>>>(gate->flags, gate->dev_seq, g, dev.status);
    if (cudaGetLastError() != cudaSuccess) return QMV_E_CUDA;
    n_before = 0;
  }
  for (int i = 0; i < n_before; ++i)
    if (copy(before[i], s) != cudaSuccess) return QMV_E_CUDA;
  for (int i = 0; i < n_groups; ++i) {
    const qmv_group& g = groups[i];
    const int st = qmv_matvec_grouped(g.wtype, g.scale_dtype, g.x_dtype, g.batch, g.problems, g.n, g.flags, s);
    if (st != QMV_OK) return st;
  }
  for (int i = 0; i < n_after; ++i)
    if (copy(after[i], s) != cudaSuccess) return QMV_E_CUDA;
  if (gate != nullptr) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, step_done_kernel, gate->flags + 1, gate->dev_seq) != cudaSuccess) return QMV_E_CUDA;
  }
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

// Frees what a step holds besides its graph (the private stream, its workspaces, the gate's
// counters).
void release_parts(cudaStream_t cap, int device, unsigned long long* flags, unsigned long long* dev_seq) {
  discard(cap, device);
  if (flags != nullptr) cudaFreeHost(flags);
  if (dev_seq != nullptr) cudaFree(dev_seq);
}

int create(const qmv_copy* before, int n_before, const qmv_group* groups, int n_groups, const qmv_copy* after,
           int n_after, bool gated, qmv_step** step) {
  if (step == nullptr) return QMV_E_ARG;
  *step = nullptr;
  if (!copies_ok(before, n_before) || !copies_ok(after, n_after)) return QMV_E_ARG;
  if (n_groups < 0 || (n_groups > 0 && groups == nullptr)) return QMV_E_ARG;
  if (gated) {
    GateCopies g;
    if (!gate_copies(before, n_before, &g)) return QMV_E_ARG;
  }
  qmv::DeviceInfo dev;
  if (qmv::current_device_info(&dev) != cudaSuccess) return QMV_E_CUDA;
  // the step as it will be kept (graph parts filled in below)
  qmv_step proto{};
  proto.device = dev.device;
  proto.gated = gated;
  if (gated) {
    void* h = nullptr;
    if (cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) return QMV_E_CUDA;
    proto.flags = static_cast<unsigned long long*>(h);
    proto.flags[0] = proto.flags[1] = 0;
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess || d != h ||
        cudaMalloc(&d, sizeof(unsigned long long)) != cudaSuccess) {
      cudaFreeHost(h);
      return QMV_E_CUDA;
    }
    proto.dev_seq = static_cast<unsigned long long*>(d);
    if (cudaMemset(proto.dev_seq, 0, sizeof(unsigned long long)) != cudaSuccess) {
      cudaFreeHost(h);
      cudaFree(d);
      return QMV_E_CUDA;
    }
  }
  cudaStream_t cap = nullptr;
  if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) {
    if (gated) {
      cudaFreeHost(proto.flags);
      cudaFree(proto.dev_seq);
    }
    return QMV_E_CUDA;
  }
  proto.cap = cap;
  if (qmv::prepare_stream_workspaces(dev, cap) != cudaSuccess) {
    release_parts(cap, dev.device, proto.flags, proto.dev_seq);
    return QMV_E_CUDA;
  }
  // the eager run (kernel attributes, checks of every argument); a gated one is opened first
  if (gated) __atomic_store_n(&proto.flags[0], 1ull, __ATOMIC_RELEASE);
  int st = enqueue(before, n_before, groups, n_groups, after, n_after, cap, gated ? &proto : nullptr);
  if (st == QMV_OK && cudaStreamSynchronize(cap) != cudaSuccess) st = QMV_E_CUDA;
  if (st == QMV_OK && gated && __atomic_load_n(&proto.flags[1], __ATOMIC_ACQUIRE) != 1ull) st = QMV_E_CUDA;
  if (st != QMV_OK) {
    release_parts(cap, dev.device, proto.flags, proto.dev_seq);
    return st;
  }
  proto.submitted = proto.opened = gated ? 1 : 0;
  // the recording
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    release_parts(cap, dev.device, proto.flags, proto.dev_seq);
    return QMV_E_CUDA;
  }
  st = enqueue(before, n_before, groups, n_groups, after, n_after, cap, gated ? &proto : nullptr);
  cudaGraph_t graph = nullptr;
  const cudaError_t end = cudaStreamEndCapture(cap, &graph);  // always ends the capture
  cudaGraphExec_t exec = nullptr;
  if (st == QMV_OK && (end != cudaSuccess || graph == nullptr)) st = QMV_E_CUDA;
  if (st == QMV_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) st = QMV_E_CUDA;
  qmv_step* s = nullptr;
  if (st == QMV_OK) {
    proto.graph = graph;
    proto.exec = exec;
    s = new (std::nothrow) qmv_step(proto);
    if (s == nullptr) st = QMV_E_CUDA;
  }
  if (st != QMV_OK) {
    if (exec != nullptr) cudaGraphExecDestroy(exec);
    if (graph != nullptr) cudaGraphDestroy(graph);
    release_parts(cap, dev.device, proto.flags, proto.dev_seq);
    return st;
  }
  *step = s;
  return QMV_OK;
}

// The host's wait for a gated step's opened runs: spins on the done count (acquire), up to
// timeout_us microseconds (10 s when <= 0).
int wait_done(qmv_step* step, long long timeout_us) {
  const unsigned long long want = step->opened;
  const auto limit = std::chrono::microseconds(timeout_us > 0 ? timeout_us : 10000000LL);
  const auto t0 = std::chrono::steady_clock::now();
  for (unsigned spin = 0;; ++spin) {
    if (__atomic_load_n(&step->flags[1], __ATOMIC_ACQUIRE) >= want) return QMV_OK;
    if ((spin & 255u) == 255u && std::chrono::steady_clock::now() - t0 > limit) return QMV_E_TIMEOUT;
  }
}

}  // namespace

extern "C" {

int qmv_step_create(const qmv_copy* before, int n_before, const qmv_group* groups, int n_groups,
                    const qmv_copy* after, int n_after, qmv_step** step) {
  return create(before, n_before, groups, n_groups, after, n_after, false, step);
}

int qmv_step_create_gated(const qmv_copy* before, int n_before, const qmv_group* groups, int n_groups,
                          const qmv_copy* after, int n_after, qmv_step** step) {
  return create(before, n_before, groups, n_groups, after, n_after, true, step);
}

int qmv_step_run(qmv_step* step, cudaStream_t stream) {
  if (step == nullptr) return QMV_E_ARG;
  if (cudaGraphLaunch(step->exec, stream) != cudaSuccess) return QMV_E_CUDA;
  ++step->submitted;
  return QMV_OK;
}

int qmv_step_open(qmv_step* step) {
  if (step == nullptr || !step->gated || step->opened >= step->submitted) return QMV_E_ARG;
  ++step->opened;
  __atomic_store_n(&step->flags[0], step->opened, __ATOMIC_RELEASE);
  return QMV_OK;
}

int qmv_step_wait(qmv_step* step, long long timeout_us) {
  if (step == nullptr || !step->gated) return QMV_E_ARG;
  return wait_done(step, timeout_us);
}

int qmv_step_open_wait(qmv_step* step, qmv_step* next, cudaStream_t stream, long long timeout_us) {
  if (step == nullptr || !step->gated || (next != nullptr && !next->gated)) return QMV_E_ARG;
  int st = qmv_step_open(step);
  if (st != QMV_OK) return st;
  if (next != nullptr && (st = qmv_step_run(next, stream)) != QMV_OK) return st;
  return wait_done(step, timeout_us);
}

int qmv_step_run_wait(qmv_step* step, cudaStream_t stream) {
  if (step == nullptr) return QMV_E_ARG;
  if (cudaGraphLaunch(step->exec, stream) != cudaSuccess) return QMV_E_CUDA;
  ++step->submitted;
  if (step->gated) {
    const int st = qmv_step_open(step);
    return st != QMV_OK ? st : wait_done(step, 0);
  }
  return cudaStreamSynchronize(stream) == cudaSuccess ? QMV_OK : QMV_E_CUDA;
}

int qmv_step_destroy(qmv_step* step) {
  if (step == nullptr) return QMV_OK;
  if (step->gated && step->opened < step->submitted) {
    step->opened = step->submitted;  // let every enqueued run through its gate
    __atomic_store_n(&step->flags[0], step->opened, __ATOMIC_RELEASE);
  }
  int st = cudaDeviceSynchronize() == cudaSuccess ? QMV_OK : QMV_E_CUDA;
  if (cudaGraphExecDestroy(step->exec) != cudaSuccess) st = QMV_E_CUDA;
  if (cudaGraphDestroy(step->graph) != cudaSuccess) st = QMV_E_CUDA;
  if (qmv::release_stream_workspaces(step->device, step->cap) != cudaSuccess) st = QMV_E_CUDA;
  if (cudaStreamDestroy(step->cap) != cudaSuccess) st = QMV_E_CUDA;
  if (step->gated) {
    if (cudaFreeHost(step->flags) != cudaSuccess) st = QMV_E_CUDA;
    if (cudaFree(step->dev_seq) != cudaSuccess) st = QMV_E_CUDA;
  }
  delete step;
  return st;
}

}  // extern "C"
