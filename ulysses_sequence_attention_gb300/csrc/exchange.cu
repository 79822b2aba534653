// exchange.cu — the two Ulysses all-to-alls, as HBM -> HBM permutations on one GPU.
//
// HF blog "Ulysses Sequence Parallelism: Training with Million-Token Contexts",
// algorithm steps 3 and 5. The first all-to-all leaves every rank with all
// sequence positions for a subset of the heads. The second one reverses it.
// The Transformers guide (section "Ulysses 序列并行的核心原理", 2-GPU diagram)
// fixes the layout: contiguous token blocks before, contiguous head blocks after.
//
// Each (rank, token, batch) row of a head shard is one contiguous run of
// Hh*hs elements in both layouts. The kernels move whole 16-byte vectors.
// Every thread keeps UNROLL independent loads in flight before it stores, so
// an SM holds enough bytes in flight to saturate HBM. The grid is a whole
// number of waves over the device's SMs. Index arithmetic uses multiply-shift
// division by invariant integers (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994).
#include "internal.cuh"

namespace uly {
namespace {

// q = x / d for every 32-bit x, via a 33-bit magic number split as (m, s).
struct FastDiv {
  uint32_t d, m, s;
  FastDiv() = default;
  explicit FastDiv(uint32_t div) : d(div) {
    s = 0;
    while ((1ull << s) < div) ++s;
    m = (uint32_t)(((1ull << 32) * ((1ull << s) - div)) / div + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t x) const {
    return (uint32_t)(((uint64_t)__umulhi(x, m) + x) >> s);
  }
  __device__ __forceinline__ void divmod(uint32_t x, uint32_t& q, uint32_t& r) const {
    q = div(x);
    r = x - q * d;
  }
};

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct S2HArgs {
  RankPtrs src;        // P sequence shards [n][bs][H][hs]
  RankPtrsMut dst;     // P head shards [sl][bs][Hh][hs]
  uint32_t total;      // vectors over all destination shards
  FastDiv per_rank;    // vectors per destination shard
  FastDiv row_vecs;    // vectors per (t, b) row of a head shard = Hh*hs*esize/16
  FastDiv bs;          // batch
  FastDiv n;           // tokens per sequence shard
  uint32_t src_row_vecs;  // vectors per (t', b) row of a sequence shard = H*hs*esize/16
  uint32_t head_vecs;     // vectors per head = hs*esize/16
  int H, P, replicated;
};

// Vector g of the destination (head shards) of one seq->head exchange: its
// source address, and its destination in *out.
__device__ __forceinline__ const uint4* s2h_vector(const S2HArgs& a, uint32_t g, uint4** out) {
  uint32_t r, rem, row, v, t, b, s, tl;
  a.per_rank.divmod(g, r, rem);
  a.row_vecs.divmod(rem, row, v);
  a.bs.divmod(row, t, b);
  a.n.divmod(t, s, tl);
  // First head of rank r's block (replicated: its single head r*H/P).
  const uint32_t h0 = a.replicated ? (r * (uint32_t)a.H) / (uint32_t)a.P : r * a.row_vecs.d / a.head_vecs;
  *out = reinterpret_cast<uint4*>(a.dst.p[r]) + rem;
  return reinterpret_cast<const uint4*>(a.src.p[s]) + (size_t)(tl * a.bs.d + b) * a.src_row_vecs +
         (size_t)h0 * a.head_vecs + v;
}

__global__ void __launch_bounds__(kThreads) seq_to_head_kernel(const __grid_constant__ S2HArgs a) {
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < a.total; base += stride * kUnroll) {
    uint4 val[kUnroll];
    uint4* out[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t g = base + u * stride;
      out[u] = nullptr;
      if (g < a.total) val[u] = __ldcs(s2h_vector(a, g, &out[u]));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (out[u]) *out[u] = val[u];
  }
}

// Up to three exchanges in one launch (the layer's Q, K and V): the vector
// index runs over the tensors one after the other, end[k] being the
// cumulative vector count through tensor k.
struct S2HMulti {
  S2HArgs t[3];
  uint32_t end[3];
  int count;
};

__global__ void __launch_bounds__(kThreads) seq_to_head_multi_kernel(const __grid_constant__ S2HMulti m) {
  const uint32_t total = m.end[m.count - 1];
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < total; base += stride * kUnroll) {
    uint4 val[kUnroll];
    uint4* out[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t g = base + u * stride;
      out[u] = nullptr;
      if (g < total) {
        const int k = g < m.end[0] ? 0 : (g < m.end[1] ? 1 : 2);
        val[u] = __ldcs(s2h_vector(m.t[k], k ? g - m.end[k - 1] : g, &out[u]));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (out[u]) *out[u] = val[u];
  }
}

struct H2SArgs {
  RankPtrs src;        // P head shards [sl][bs][Hh][hs]
  RankPtrsMut dst;     // P sequence shards [n][bs][H][hs]
  uint32_t total;      // vectors over all destination shards
  FastDiv per_shard;   // vectors per sequence shard
  FastDiv row_vecs;    // vectors per (t', b) row of a sequence shard = H*hs*esize/16
  FastDiv bs;
  FastDiv block_vecs;  // vectors per rank block of heads = Hh*hs*esize/16
  uint32_t n;          // tokens per sequence shard
};

// Vector g of the destination (sequence shards) of one head->seq exchange.
__device__ __forceinline__ const uint4* h2s_vector(const H2SArgs& a, uint32_t g, uint4** out) {
  uint32_t s, rem, row, v, tl, b, r, w;
  a.per_shard.divmod(g, s, rem);
  a.row_vecs.divmod(rem, row, v);
  a.bs.divmod(row, tl, b);
  a.block_vecs.divmod(v, r, w);
  const uint32_t t = s * a.n + tl;
  *out = reinterpret_cast<uint4*>(a.dst.p[s]) + rem;
  return reinterpret_cast<const uint4*>(a.src.p[r]) + (size_t)(t * a.bs.d + b) * a.block_vecs.d + w;
}

__global__ void __launch_bounds__(kThreads) head_to_seq_kernel(const __grid_constant__ H2SArgs a) {
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < a.total; base += stride * kUnroll) {
    uint4 val[kUnroll];
    uint4* out[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t g = base + u * stride;
      out[u] = nullptr;
      if (g < a.total) val[u] = __ldcs(h2s_vector(a, g, &out[u]));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (out[u]) *out[u] = val[u];
  }
}

// Up to three head->seq exchanges in one launch (dQ, dK and dV).
struct H2SMulti {
  H2SArgs t[3];
  uint32_t end[3];
  int count;
};

__global__ void __launch_bounds__(kThreads) head_to_seq_multi_kernel(const __grid_constant__ H2SMulti m) {
  const uint32_t total = m.end[m.count - 1];
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t base = blockIdx.x * kThreads + threadIdx.x; base < total; base += stride * kUnroll) {
    uint4 val[kUnroll];
    uint4* out[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t g = base + u * stride;
      out[u] = nullptr;
      if (g < total) {
        const int k = g < m.end[0] ? 0 : (g < m.end[1] ? 1 : 2);
        val[u] = __ldcs(h2s_vector(m.t[k], k ? g - m.end[k - 1] : g, &out[u]));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (out[u]) *out[u] = val[u];
  }
}

// Replicated kv heads (P > H): the gradient of head h is the sum of the
// P/H replicas held by ranks [h*P/H, (h+1)*P/H). One thread per element.
template <typename T>
__global__ void __launch_bounds__(kThreads) head_to_seq_sum_kernel(RankPtrs src, RankPtrsMut dst,
                                                                   uint32_t total, FastDiv per_shard,
                                                                   FastDiv row_elems, FastDiv bs,
                                                                   FastDiv hs, uint32_t n, int reps) {
  for (uint32_t g = blockIdx.x * kThreads + threadIdx.x; g < total; g += gridDim.x * kThreads) {
    uint32_t s, rem, row, e, tl, b, h, d;
    per_shard.divmod(g, s, rem);
    row_elems.divmod(rem, row, e);
    bs.divmod(row, tl, b);
    hs.divmod(e, h, d);
    const uint32_t t = s * n + tl;
    float acc = 0.f;
    for (int k = 0; k < reps; ++k) {
      const T* p = reinterpret_cast<const T*>(src.p[h * reps + k]);
      acc += to_f32<T>(p[(size_t)(t * bs.d + b) * hs.d + d]);
    }
    reinterpret_cast<T*>(dst.p[s])[rem] = from_f32<T>(acc);
  }
}

int grid_for(uint64_t items_per_thread_block) {
  uint64_t g = (items_per_thread_block + (uint64_t)kThreads * kUnroll - 1) / ((uint64_t)kThreads * kUnroll);
  const uint64_t cap = (uint64_t)device_sm_count() * 8;  // 8 resident 256-thread blocks per SM
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

// Arguments of one seq->head exchange of an nheads-head tensor; its vector count in *total.
static int make_s2h(const Layer& L, int nheads, const void* const* src, void* const* dst, S2HArgs& a,
                    uint64_t* total) {
  const int H = nheads;
  const bool replicated = (H % L.P) != 0;
  const int Hh = replicated ? 1 : H / L.P;
  const uint32_t head_vecs = (uint32_t)(L.hs * L.esize() / 16);
  const uint64_t per_rank = (uint64_t)L.sl * L.bs * Hh * head_vecs;
  *total = per_rank * L.P;
  if (*total >= (1ull << 32)) return ULYSSES_ERR_UNSUPPORTED;
  for (int r = 0; r < L.P; ++r) {
    a.src.p[r] = src[r];
    a.dst.p[r] = dst[r];
  }
  a.total = (uint32_t)*total;
  a.per_rank = FastDiv((uint32_t)per_rank);
  a.row_vecs = FastDiv((uint32_t)Hh * head_vecs);
  a.bs = FastDiv((uint32_t)L.bs);
  a.n = FastDiv((uint32_t)L.n());
  a.src_row_vecs = (uint32_t)H * head_vecs;
  a.head_vecs = head_vecs;
  a.H = H;
  a.P = L.P;
  a.replicated = replicated ? 1 : 0;
  return ULYSSES_OK;
}

// Arguments of one head->seq exchange (nheads % P == 0); its vector count in *total.
static int make_h2s(const Layer& L, int nheads, const void* const* src, void* const* dst, H2SArgs& a,
                    uint64_t* total) {
  const int H = nheads;
  const uint64_t n = (uint64_t)L.n();
  const int Hh = H / L.P;
  const uint32_t head_vecs = (uint32_t)(L.hs * L.esize() / 16);
  const uint64_t per_shard = n * L.bs * H * head_vecs;
  *total = per_shard * L.P;
  if (*total >= (1ull << 32)) return ULYSSES_ERR_UNSUPPORTED;
  for (int r = 0; r < L.P; ++r) {
    a.src.p[r] = src[r];
    a.dst.p[r] = dst[r];
  }
  a.total = (uint32_t)*total;
  a.per_shard = FastDiv((uint32_t)per_shard);
  a.row_vecs = FastDiv((uint32_t)H * head_vecs);
  a.bs = FastDiv((uint32_t)L.bs);
  a.block_vecs = FastDiv((uint32_t)Hh * head_vecs);
  a.n = (uint32_t)n;
  return ULYSSES_OK;
}

int launch_seq_to_head(const Layer& L, int nheads, const void* const* src, void* const* dst,
                       cudaStream_t stream) {
  S2HArgs a;
  uint64_t total = 0;
  const int st = make_s2h(L, nheads, src, dst, a, &total);
  if (st != ULYSSES_OK) return st;
  Timed t(L.timing, ULYSSES_KERNEL_SEQ_TO_HEAD, stream);
  seq_to_head_kernel<<<grid_for(total), kThreads, 0, stream>>>(a);
  t.done();
  count_launches(1);
  return cuda_status(cudaGetLastError());
}

int launch_seq_to_head_multi(const Layer& L, int count, const int* nheads, const void* const* const* src,
                             void* const* const* dst, cudaStream_t stream) {
  S2HMulti m;
  uint64_t end = 0;
  m.count = count;
  for (int k = 0; k < count; ++k) {
    uint64_t total = 0;
    const int st = make_s2h(L, nheads[k], src[k], dst[k], m.t[k], &total);
    if (st != ULYSSES_OK) return st;
    end += total;
    if (end >= (1ull << 32)) return ULYSSES_ERR_UNSUPPORTED;
    m.end[k] = (uint32_t)end;
  }
  Timed t(L.timing, ULYSSES_KERNEL_SEQ_TO_HEAD, stream);
  seq_to_head_multi_kernel<<<grid_for(end), kThreads, 0, stream>>>(m);
  t.done();
  count_launches(1);
  return cuda_status(cudaGetLastError());
}

int launch_head_to_seq(const Layer& L, int nheads, const void* const* src, void* const* dst,
                       cudaStream_t stream) {
  const int H = nheads;
  const uint64_t n = (uint64_t)L.n();
  if (H % L.P != 0) {
    // Replicated kv heads: sum the replicas of each head's gradient.
    const int reps = L.P / H;
    const uint64_t per_shard = n * L.bs * H * L.hs;
    const uint64_t total = per_shard * L.P;
    if (total >= (1ull << 32)) return ULYSSES_ERR_UNSUPPORTED;
    RankPtrs s;
    RankPtrsMut d;
    for (int r = 0; r < L.P; ++r) {
      s.p[r] = src[r];
      d.p[r] = dst[r];
    }
    uint64_t g = (total + kThreads - 1) / kThreads;
    if (g > (uint64_t)device_sm_count() * 8) g = (uint64_t)device_sm_count() * 8;
    Timed t(L.timing, ULYSSES_KERNEL_HEAD_TO_SEQ, stream);
    if (L.dtype == ULYSSES_BF16)
      head_to_seq_sum_kernel<__nv_bfloat16><<<(int)g, kThreads, 0, stream>>>(
          s, d, (uint32_t)total, FastDiv((uint32_t)per_shard), FastDiv((uint32_t)(H * L.hs)),
          FastDiv((uint32_t)L.bs), FastDiv((uint32_t)L.hs), (uint32_t)n, reps);
    else
      head_to_seq_sum_kernel<float><<<(int)g, kThreads, 0, stream>>>(
          s, d, (uint32_t)total, FastDiv((uint32_t)per_shard), FastDiv((uint32_t)(H * L.hs)),
          FastDiv((uint32_t)L.bs), FastDiv((uint32_t)L.hs), (uint32_t)n, reps);
    t.done();
    count_launches(1);
    return cuda_status(cudaGetLastError());
  }
  H2SArgs a;
  uint64_t total = 0;
  const int st = make_h2s(L, H, src, dst, a, &total);
  if (st != ULYSSES_OK) return st;
  Timed t(L.timing, ULYSSES_KERNEL_HEAD_TO_SEQ, stream);
  head_to_seq_kernel<<<grid_for(total), kThreads, 0, stream>>>(a);
  t.done();
  count_launches(1);
  return cuda_status(cudaGetLastError());
}

int launch_head_to_seq_multi(const Layer& L, int count, const int* nheads, const void* const* const* src,
                             void* const* const* dst, cudaStream_t stream) {
  for (int k = 0; k < count; ++k)
    if (nheads[k] % L.P != 0) {
      // Replicated kv heads need the replica sum: one launch per tensor.
      for (int j = 0; j < count; ++j) {
        const int st = launch_head_to_seq(L, nheads[j], src[j], dst[j], stream);
        if (st != ULYSSES_OK) return st;
      }
      return ULYSSES_OK;
    }
  H2SMulti m;
  uint64_t end = 0;
  m.count = count;
  for (int k = 0; k < count; ++k) {
    uint64_t total = 0;
    const int st = make_h2s(L, nheads[k], src[k], dst[k], m.t[k], &total);
    if (st != ULYSSES_OK) return st;
    end += total;
    if (end >= (1ull << 32)) return ULYSSES_ERR_UNSUPPORTED;
    m.end[k] = (uint32_t)end;
  }
  Timed t(L.timing, ULYSSES_KERNEL_HEAD_TO_SEQ, stream);
  head_to_seq_multi_kernel<<<grid_for(end), kThreads, 0, stream>>>(m);
  t.done();
  count_launches(1);
  return cuda_status(cudaGetLastError());
}

}  // namespace uly
