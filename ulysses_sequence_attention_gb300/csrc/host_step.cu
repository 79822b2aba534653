// host_step.cu — training steps of the layer from host memory, with the
// host<->device copies overlapped with the compute of neighbouring steps.
//
// A step is what a training loop feeds the layer: the sequence shards of Q, K,
// V and dO arrive from the host, the forward and backward run (the exchanges
// fused into the attention kernels, ulysses_layer_fwd / _bwd), and O, dQ, dK,
// dV go back to the host. In the pages' training loop the data loader hands
// each rank its sequence shard (ALST guide, section 2.2, the DataLoader
// adapter with its CPU prefetch buffer); here the P shards of a step are host
// buffers.
//
// Streams: the caller's stream runs the kernels; the handle owns one stream for
// host->device and one for device->host copies. Two slots of device buffers
// let step i+1's inputs travel while step i computes, and step i's outputs
// travel while step i+1 computes. Events order every reuse of a slot:
//   H2D into slot s        waits for the last compute on slot s (it reads the inputs);
//   the forward on slot s  waits for its Q, K, V and for the last D2H out of slot s;
//   the backward           waits for dO;
//   D2H of O               waits for the forward (it overlaps the backward);
//   D2H of dQ, dK, dV      waits for the backward.
// LSE and the workspace are shared by the slots: all kernels run on one stream.
#include "internal.cuh"

namespace uly {

void destroy_host_pipe(Layer& L) {
  Layer::HostPipe& p = L.pipe;
  for (int s = 0; s < 2; ++s) {
    for (cudaEvent_t e : {p.qkv_in[s], p.do_in[s], p.o_done[s], p.computed[s], p.out_copied[s]})
      if (e) cudaEventDestroy(e);
  }
  for (cudaEvent_t e : {p.fork, p.h2d_tail, p.d2h_tail})
    if (e) cudaEventDestroy(e);
  if (p.h2d) cudaStreamDestroy(p.h2d);
  if (p.d2h) cudaStreamDestroy(p.d2h);
  p = Layer::HostPipe();
}

static int ensure_pipe(Layer& L) {
  Layer::HostPipe& p = L.pipe;
  if (p.ready) return ULYSSES_OK;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return ULYSSES_ERR_CUDA;
  if (cur != L.device && cudaSetDevice(L.device) != cudaSuccess) return ULYSSES_ERR_CUDA;
  cudaError_t e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking);
  for (int s = 0; s < 2 && e == cudaSuccess; ++s) {
    for (cudaEvent_t* ev : {&p.qkv_in[s], &p.do_in[s], &p.o_done[s], &p.computed[s], &p.out_copied[s]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  }
  for (cudaEvent_t* ev : {&p.fork, &p.h2d_tail, &p.d2h_tail})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (cur != L.device) cudaSetDevice(cur);
  if (e != cudaSuccess) {
    destroy_host_pipe(L);
    return ULYSSES_ERR_CUDA;
  }
  p.ready = true;
  return ULYSSES_OK;
}

// Copies P shards of `bytes` each, src[r] -> dst[r], on stream s.
static cudaError_t copy_shards(void* const* dst, const void* const* src, int P, size_t bytes, cudaMemcpyKind kind,
                               cudaStream_t s) {
  for (int r = 0; r < P; ++r) {
    const cudaError_t e = cudaMemcpyAsync(dst[r], src[r], bytes, kind, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace uly

using uly::Layer;

extern "C" {

int ulysses_host_begin(ulysses_t h, void* stream) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (!uly::fused_supported(*L) && !L->empty()) return ULYSSES_ERR_UNSUPPORTED;
  int st = uly::ensure_pipe(*L);
  if (st != ULYSSES_OK) return st;
  Layer::HostPipe& p = L->pipe;
  cudaError_t e = cudaEventRecord(p.fork, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.h2d, p.fork, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.d2h, p.fork, 0);
  return uly::cuda_status(e);
}

int ulysses_host_step(ulysses_t h, int slot, const void* const* host_in, void* const* host_out, void* const* dev,
                      float* const* lse, void* workspace, void* stream) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (slot != 0 && slot != 1) return ULYSSES_ERR_INVALID_ARG;
  if (L->empty()) return ULYSSES_OK;
  if (!uly::fused_supported(*L)) return ULYSSES_ERR_UNSUPPORTED;
  const int P = L->P;
  if (!host_in || !host_out || !dev || !lse || !workspace) return ULYSSES_ERR_INVALID_ARG;
  for (int i = 0; i < 4 * P; ++i)
    if (!host_in[i] || !host_out[i]) return ULYSSES_ERR_INVALID_ARG;
  for (int i = 0; i < 8 * P; ++i) {
    if (!dev[i]) return ULYSSES_ERR_INVALID_ARG;
    if (((uintptr_t)dev[i]) & 15u) return ULYSSES_ERR_ALIGNMENT;
  }
  for (int r = 0; r < P; ++r) {
    if (!lse[r]) return ULYSSES_ERR_INVALID_ARG;
    if (((uintptr_t)lse[r]) & 15u) return ULYSSES_ERR_ALIGNMENT;
  }
  if (((uintptr_t)workspace) & 15u) return ULYSSES_ERR_ALIGNMENT;
  int st = uly::ensure_pipe(*L);
  if (st != ULYSSES_OK) return st;
  Layer::HostPipe& p = L->pipe;
  cudaStream_t cs = (cudaStream_t)stream;

  const size_t row = (size_t)L->bs * L->hs * L->esize();
  const size_t nq = (size_t)L->n() * L->hc * row;    // bytes of a Q/O/dO/dQ shard
  const size_t nk = (size_t)L->n() * L->hkv * row;   // bytes of a K/V/dK/dV shard
  void* const* dq_ = dev;            // device Q
  void* const* dk_ = dev + P;        // device K
  void* const* dv_ = dev + 2 * P;    // device V
  void* const* ddo = dev + 3 * P;    // device dO
  void* const* dO_ = dev + 4 * P;    // device O
  void* const* gq = dev + 5 * P;     // device dQ
  void* const* gk = dev + 6 * P;     // device dK
  void* const* gv = dev + 7 * P;     // device dV

  // 1. Inputs in, once the last compute on this slot has read its inputs.
  cudaError_t e = cudaStreamWaitEvent(p.h2d, p.computed[slot], 0);
  if (e == cudaSuccess) e = uly::copy_shards(dq_, host_in, P, nq, cudaMemcpyHostToDevice, p.h2d);
  if (e == cudaSuccess) e = uly::copy_shards(dk_, host_in + P, P, nk, cudaMemcpyHostToDevice, p.h2d);
  if (e == cudaSuccess) e = uly::copy_shards(dv_, host_in + 2 * P, P, nk, cudaMemcpyHostToDevice, p.h2d);
  if (e == cudaSuccess) e = cudaEventRecord(p.qkv_in[slot], p.h2d);
  if (e == cudaSuccess) e = uly::copy_shards(ddo, host_in + 3 * P, P, nq, cudaMemcpyHostToDevice, p.h2d);
  if (e == cudaSuccess) e = cudaEventRecord(p.do_in[slot], p.h2d);
  if (e != cudaSuccess) return ULYSSES_ERR_CUDA;

  // 2. Forward, once Q, K, V are in and the last outputs of this slot are out.
  e = cudaStreamWaitEvent(cs, p.qkv_in[slot], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, p.out_copied[slot], 0);
  if (e != cudaSuccess) return ULYSSES_ERR_CUDA;
  st = ulysses_layer_fwd(h, (const void* const*)dq_, (const void* const*)dk_, (const void* const*)dv_, dO_, lse,
                         stream);
  if (st != ULYSSES_OK) return st;
  e = cudaEventRecord(p.o_done[slot], cs);
  // 3. Backward, once dO is in.
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, p.do_in[slot], 0);
  if (e != cudaSuccess) return ULYSSES_ERR_CUDA;
  st = ulysses_layer_bwd(h, (const void* const*)dq_, (const void* const*)dk_, (const void* const*)dv_,
                         (const void* const*)dO_, (const void* const*)ddo, (const float* const*)lse, gq, gk, gv,
                         workspace, stream);
  if (st != ULYSSES_OK) return st;
  e = cudaEventRecord(p.computed[slot], cs);

  // 4. Outputs out: O while the backward runs, then dQ, dK, dV.
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.d2h, p.o_done[slot], 0);
  if (e == cudaSuccess) e = uly::copy_shards(host_out, (const void* const*)dO_, P, nq, cudaMemcpyDeviceToHost, p.d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.d2h, p.computed[slot], 0);
  if (e == cudaSuccess)
    e = uly::copy_shards(host_out + P, (const void* const*)gq, P, nq, cudaMemcpyDeviceToHost, p.d2h);
  if (e == cudaSuccess)
    e = uly::copy_shards(host_out + 2 * P, (const void* const*)gk, P, nk, cudaMemcpyDeviceToHost, p.d2h);
  if (e == cudaSuccess)
    e = uly::copy_shards(host_out + 3 * P, (const void* const*)gv, P, nk, cudaMemcpyDeviceToHost, p.d2h);
  if (e == cudaSuccess) e = cudaEventRecord(p.out_copied[slot], p.d2h);
  return uly::cuda_status(e);
}

int ulysses_host_end(ulysses_t h, void* stream) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (!L->pipe.ready) return ULYSSES_OK;  // no step was ever enqueued
  Layer::HostPipe& p = L->pipe;
  cudaError_t e = cudaEventRecord(p.h2d_tail, p.h2d);
  if (e == cudaSuccess) e = cudaEventRecord(p.d2h_tail, p.d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent((cudaStream_t)stream, p.h2d_tail, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent((cudaStream_t)stream, p.d2h_tail, 0);
  return uly::cuda_status(e);
}

}  // extern "C"
