// internal.cuh — shared host/device definitions of the Ulysses layer library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <atomic>
#include <vector>

#include "../../include/ulysses.h"

namespace uly {

// Bits of the device status word (see ulysses_get_status).
enum : unsigned {
  STATUS_TIMEOUT = 1u,
};

// Per-kernel device time of one handle (ulysses_timing_enable / _read). Each
// timed launch is bracketed by two events on its stream; the records wait in
// `pending` until a read (or a full queue) synchronises them.
struct Timing {
  struct Rec {
    int kernel;
    cudaEvent_t a, b;
  };
  bool on = false;
  bool failed = false;
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> spare;
  double total_ms[ULYSSES_KERNEL_COUNT] = {};
  int64_t launches[ULYSSES_KERNEL_COUNT] = {};

  Timing() = default;
  Timing(const Timing&) = delete;
  Timing& operator=(const Timing&) = delete;

  cudaEvent_t take() {
    if (!spare.empty()) {
      cudaEvent_t e = spare.back();
      spare.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
      failed = true;
      return nullptr;
    }
    return e;
  }
  // Called right before a launch: the start event, or null when timing is off.
  cudaEvent_t begin(cudaStream_t s) {
    if (!on) return nullptr;
    cudaEvent_t a = take();
    if (a && cudaEventRecord(a, s) != cudaSuccess) {
      failed = true;
      spare.push_back(a);
      return nullptr;
    }
    return a;
  }
  // Called right after the launch with what begin returned.
  void end(int kernel, cudaEvent_t a, cudaStream_t s) {
    if (!a) return;
    cudaEvent_t b = take();
    if (!b || cudaEventRecord(b, s) != cudaSuccess) {
      failed = true;
      spare.push_back(a);
      if (b) spare.push_back(b);
      return;
    }
    pending.push_back({kernel, a, b});
    if (pending.size() >= 8192) drain(4096);
  }
  // Folds the oldest n pending records into the totals (waits for them).
  void drain(size_t n) {
    n = n < pending.size() ? n : pending.size();
    for (size_t i = 0; i < n; ++i) {
      const Rec& r = pending[i];
      float ms = 0.f;
      if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
        failed = true;
      total_ms[r.kernel] += ms;
      launches[r.kernel] += 1;
      spare.push_back(r.a);
      spare.push_back(r.b);
    }
    pending.erase(pending.begin(), pending.begin() + (long)n);
  }
  void reset() {
    drain(pending.size());
    for (int k = 0; k < ULYSSES_KERNEL_COUNT; ++k) {
      total_ms[k] = 0.0;
      launches[k] = 0;
    }
    failed = false;
  }
  ~Timing() {
    for (const Rec& r : pending) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
    for (cudaEvent_t e : spare) cudaEventDestroy(e);
  }
};

// Brackets one kernel launch: `Timed t(L, ULYSSES_KERNEL_X, s); kernel<<<...>>>(...); t.done();`
struct Timed {
  Timing& T;
  int kernel;
  cudaStream_t s;
  cudaEvent_t a;
  Timed(Timing& T_, int k, cudaStream_t s_) : T(T_), kernel(k), s(s_), a(T_.begin(s_)) {}
  void done() { T.end(kernel, a, s); }
};

struct Layer {
  int64_t sl = 0, bs = 0;
  int hc = 0, hkv = 0, hs = 0, P = 0, causal = 1, dtype = ULYSSES_BF16;
  int Hq = 0;       // query heads per rank (hc / P)
  int Hk = 0;       // kv heads per rank (hkv / P, or 1 when replicated)
  int ndoc = 1;
  int64_t cap_sl = 0;                 // device tables hold sequences up to cap_sl tokens
  int cap_docs = 1;                   // ... in up to cap_docs documents
  std::vector<int32_t> doc_offsets;   // host copy, ndoc + 1 entries
  int32_t* d_doc_offsets = nullptr;   // device copy, ndoc + 1 entries
  unsigned* d_status = nullptr;       // device status word
  // The stream of the handle's latest enqueuing call: ulysses_get_status
  // reads the status word in order on it (set by every call that takes a stream).
  mutable cudaStream_t last_stream = nullptr;
  int device = 0;
  // Tensor-core path (CTA pairs): per 256-key pair tile the range of 128-row
  // query tiles that see it (dK/dV), per 256-query pair tile the range of
  // 128-key tiles it sees (forward, dQ); each with an order by work, most
  // first. Device copies.
  int2* d_kvp_range = nullptr;
  int* d_kvp_order = nullptr;
  int2* d_qp_range = nullptr;
  int* d_qp_order = nullptr;
  // Stored dS (ulysses_set_ds_budget): the dK/dV kernel also writes the bf16
  // dS of every visible (128-key tile, 128-query tile) block to the
  // workspace, and dQ = s dS K reads it back instead of recomputing S and dP.
  // Per 256-key pair tile, the index of its first block within a (rank,
  // batch, head); ds_nblk blocks per (rank, batch, head) for the current
  // sequence. The workspace reserves ds_reserved blocks per (rank, batch,
  // head) (ulysses_set_ds_budget); a backward stores dS when the current
  // sequence's ds_nblk fit.
  int* d_ds_base = nullptr;
  int64_t ds_nblk = 0;
  int64_t ds_reserved = 0;
  bool ds_fits() const { return ds_reserved > 0 && ds_nblk > 0 && ds_nblk <= ds_reserved; }
  long long timeout_cycles = 4000000000LL;  // bound of every device-side wait (~2 s)
  mutable int inject_fault = 0;             // test hook (ulysses_inject_fault), consumed by one call
  mutable Timing timing;                    // ulysses_timing_enable / ulysses_timing_read
  // Host-streaming steps (ulysses_host_begin / _step / _end): two copy
  // streams and, per device-buffer slot, the events that order its reuse.
  // Created on first use, destroyed with the handle.
  struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t qkv_in[2] = {}, do_in[2] = {}, o_done[2] = {}, computed[2] = {}, out_copied[2] = {};
    cudaEvent_t fork = nullptr, h2d_tail = nullptr, d2h_tail = nullptr;
    bool ready = false;
  } pipe;
  int64_t n() const { return sl / P; }          // tokens per sequence shard
  int esize() const { return dtype == ULYSSES_BF16 ? 2 : 4; }
  bool empty() const { return sl == 0 || bs == 0; }
};

// Per-rank pointer tables passed by value as kernel parameters.
struct RankPtrs {
  const void* p[ULYSSES_MAX_P];
};
struct RankPtrsMut {
  void* p[ULYSSES_MAX_P];
};

// Shape of the per-rank attention problem, shared by the attention kernels.
struct AttnShape {
  int sl;          // global sequence length (<= 2^30)
  int bs;
  int P;
  int Hq;          // query heads per rank
  int Hk;          // kv heads per rank
  int group;       // query heads per kv head on a rank (Hq / Hk)
  int hs;
  int causal;
  int ndoc;
  float scale;     // 1 / sqrt(hs)
  float scale_log2;  // scale * log2(e)
  const int32_t* doc_offsets;  // device, ndoc + 1
  unsigned* status;
};

AttnShape make_shape(const Layer& L);

// Host launchers (each returns a ulysses_status).
int launch_seq_to_head(const Layer& L, int nheads, const void* const* src, void* const* dst,
                       cudaStream_t s);
int launch_head_to_seq(const Layer& L, int nheads, const void* const* src, void* const* dst,
                       cudaStream_t s);
// count (<= 3) exchanges in one launch: tensor k has nheads[k] heads, P source
// pointers src[k] and P destination pointers dst[k].
int launch_seq_to_head_multi(const Layer& L, int count, const int* nheads, const void* const* const* src,
                             void* const* const* dst, cudaStream_t s);
int launch_head_to_seq_multi(const Layer& L, int count, const int* nheads, const void* const* const* src,
                             void* const* const* dst, cudaStream_t s);
int launch_attn_fwd_simt(const Layer& L, const void* const* q, const void* const* k,
                         const void* const* v, void* const* o, float* const* lse, cudaStream_t s);
int launch_attn_bwd_simt(const Layer& L, const void* const* q, const void* const* k,
                         const void* const* v, const void* const* o, const void* const* dO,
                         const float* const* lse, void* const* dq, void* const* dk,
                         void* const* dv, void* workspace, cudaStream_t s);

bool fwd_sm103_supported(const Layer& L);
// Whether the tensor-core kernels can read and write sequence shards directly
// (the exchanges fused into their TMA addressing): the bf16 hs=128 path, at
// most kMaxFusedP shards (one tensor map per shard and operand in a launch),
// shards of a whole number of 128-row tiles, and no replicated kv heads.
constexpr int kMaxFusedP = 8;
bool fused_supported(const Layer& L);
// fused: q, k, v, o are sequence shards (else head shards).
int launch_attn_fwd_sm103(Layer& L, const void* const* q, const void* const* k, const void* const* v,
                          void* const* o, float* const* lse, cudaStream_t s, bool fused = false);

void plan_pair_tiles(const Layer& L, std::vector<int2>& kv_pairs, std::vector<int>& kv_order,
                     std::vector<int2>& q_pairs, std::vector<int>& q_order);
// Stored dS blocks: base[t] = index of the first block of key pair tile t
// within a (rank, batch, head); returns the blocks per (rank, batch, head).
int64_t plan_ds_blocks(const std::vector<int2>& kv_pairs, std::vector<int>& base);
// The row planes of the tensor-core backward.
size_t bwd_sm103_workspace(const Layer& L);
// The stored-dS area that follows them (zero block + blocks) for nblk blocks
// per (rank, batch, head), and its offset in the workspace.
size_t bwd_ds_bytes(const Layer& L, int64_t nblk);
size_t bwd_ds_offset(const Layer& L);
// fused: q, k, v, o, dO, dq, dk, dv are sequence shards (else head shards).
// store_ds: the workspace holds the reserved stored-dS area and may use it
// (dS is stored when the current sequence fits it, L.ds_fits()).
int launch_attn_bwd_sm103(const Layer& L, const void* const* q, const void* const* k, const void* const* v,
                          const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
                          void* const* dk, void* const* dv, void* workspace, cudaStream_t s, bool fused = false,
                          bool store_ds = false);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA; }

// Adds n to the library-wide kernel launch counter (ulysses_launch_count).
void count_launches(int n);

// Runs a configuration step (kernel attributes) once per device: function
// attributes are per device, so a process that drives several GPUs needs it
// on each. Setting an attribute twice (two host threads racing) is harmless.
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};  // bit d: device d configured (devices >= 64: every call)
  template <class F>
  int run(F&& configure) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ULYSSES_ERR_CUDA;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return ULYSSES_OK;
    if (configure() != cudaSuccess) return ULYSSES_ERR_CUDA;
    if (bit) done.fetch_or(bit, std::memory_order_release);
    return ULYSSES_OK;
  }
};

// Workspace of the backward for the handle's capacity, with or without the
// reserved stored-dS area; the blocks per (rank, batch, head) of one
// document at capacity (the most any sequence of the handle needs).
size_t workspace_bytes(const Layer& L, bool with_ds);
int64_t ds_blocks_at_capacity(const Layer& L);
// ulysses_attn_bwd; store_ds = false keeps to the row planes of the workspace
// (the recomputing dQ), whatever the handle's dS budget.
int attn_bwd_entry(ulysses_t h, const void* const* q, const void* const* k, const void* const* v,
                   const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
                   void* const* dk, void* const* dv, void* workspace, void* stream, bool store_ds);

// Number of SMs of the current device, looked up once per device (grid
// sizing of the streaming kernels).
inline int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 1;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Looks up, and so loads, the no-alloc scratch array on the current device
// (noalloc.cu); ulysses_create calls it during set-up.
void noalloc_setup();

// Frees the host-streaming streams and events of a handle (host_step.cu).
void destroy_host_pipe(Layer& L);

}  // namespace uly

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
namespace uly {

// Document index of position t: the largest d with doc_offsets[d] <= t.
__device__ __forceinline__ int doc_of(const int32_t* offs, int ndoc, int t) {
  int lo = 0, hi = ndoc - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (offs[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Where a tile of rows [t, t + 128) of local head h of rank rl lives, for the
// TMA tensor maps of the attention kernels.
//  * Head shards (fused == 0): map rl holds rank rl's heads; coordinates are
//    (head h, row t).
//  * Sequence shards (fused != 0): the seq->head exchange read through the
//    tensor maps. Map s covers shard s, tokens [s*n, (s+1)*n) with every
//    head, so the tile is in map t / n at head rl*H + h and row t - s*n. A
//    tile never straddles two shards (n is a multiple of 128). A tile that
//    starts past the sequence (the odd CTA of a last half pair) is placed in
//    the last shard at a row >= n, where TMA reads zeros and clips stores.
struct TileLoc {
  int map, head, row;
};
__device__ __forceinline__ TileLoc locate_tile(int fused, int n, int nshards, int rl, int H, int h, int t) {
  if (!fused) return {rl, h, t};
  const int s = min(t / n, nshards - 1);
  return {s, rl * H + h, t - s * n};
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace uly
