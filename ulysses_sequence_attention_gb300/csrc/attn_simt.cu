// attn_simt.cu — exact attention forward and backward on the CUDA cores (fp32 FFMA).
//
// This is the fp32 path and the path for head sizes 32 and 64. It also runs
// bf16 inputs: every product and sum is in fp32, and only the outputs are
// rounded to bf16. It is a correctness path. The bf16 path for head size 128
// runs on the tensor cores (attn_fwd_sm103.cu, attn_bwd_sm103.cu).
//
// The equations are those of ulysses_attn_fwd / ulysses_attn_bwd. Standard
// attention per head comes from the HF blog "Ulysses Sequence Parallelism:
// Training with Million-Token Contexts", algorithm step 4. The mask comes from
// the position ids: causal, and reset at each document start (ALST guide,
// sections 2.1 and 2.2).
//
// Work split: one warp per query row (forward, dQ) or per key row (dK, dV).
// The row's own vector sits in shared memory; the lanes of the warp take 32
// keys (or queries) at a time for the dot products, then take the head
// dimension for the weighted sums.
#include "internal.cuh"

namespace uly {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerBlock = kWarps * kRowsPerWarp;

__device__ __forceinline__ void visible_keys(const AttnShape& sh, int i, int& lo, int& hi) {
  const int d = doc_of(sh.doc_offsets, sh.ndoc, i);
  lo = sh.doc_offsets[d];
  hi = sh.causal ? i : sh.doc_offsets[d + 1] - 1;
}

__device__ __forceinline__ void visible_queries(const AttnShape& sh, int j, int& lo, int& hi) {
  const int d = doc_of(sh.doc_offsets, sh.ndoc, j);
  lo = sh.causal ? j : sh.doc_offsets[d];
  hi = sh.doc_offsets[d + 1] - 1;
}

template <typename T, int HS>
__device__ __forceinline__ float dot_row(const float* __restrict__ a_smem, const T* __restrict__ b) {
  float acc = 0.f;
#pragma unroll 8
  for (int d = 0; d < HS; ++d) acc = fmaf(a_smem[d], to_f32<T>(b[d]), acc);
  return acc;
}

template <typename T, int HS>
__global__ void __launch_bounds__(kWarps * 32) attn_fwd_simt_kernel(AttnShape sh, RankPtrs qp, RankPtrs kp,
                                                                    RankPtrs vp, RankPtrsMut op,
                                                                    RankPtrsMut lp) {
  constexpr int C = HS / 32;
  __shared__ float qs[kWarps][HS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.z;
  const int b = blockIdx.y / sh.Hq, hq = blockIdx.y % sh.Hq, hk = hq / sh.group;
  const T* q = reinterpret_cast<const T*>(qp.p[r]);
  const T* k = reinterpret_cast<const T*>(kp.p[r]);
  const T* v = reinterpret_cast<const T*>(vp.p[r]);
  T* o = reinterpret_cast<T*>(op.p[r]);
  float* lse = reinterpret_cast<float*>(lp.p[r]);
  const size_t qstride = (size_t)sh.bs * sh.Hq * HS;   // between tokens
  const size_t kstride = (size_t)sh.bs * sh.Hk * HS;
  const size_t qoff = ((size_t)b * sh.Hq + hq) * HS;
  const size_t koff = ((size_t)b * sh.Hk + hk) * HS;
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int i = blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp + rr;
    if (i >= sh.sl) break;
#pragma unroll
    for (int c = 0; c < C; ++c) qs[warp][lane + 32 * c] = to_f32<T>(q[i * qstride + qoff + lane + 32 * c]);
    __syncwarp();
    int lo, hi;
    visible_keys(sh, i, lo, hi);
    float m = -INFINITY, l = 0.f, acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    for (int j0 = lo; j0 <= hi; j0 += 32) {
      const int j = j0 + lane;
      float s = -INFINITY;
      if (j <= hi) s = sh.scale * dot_row<T, HS>(qs[warp], k + j * kstride + koff);
      const float m_new = fmaxf(m, warp_max(s));
      const float alpha = expf(m - m_new);
      const float p = (j <= hi) ? expf(s - m_new) : 0.f;
      l = l * alpha + warp_sum(p);
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] *= alpha;
      const int cnt = min(32, hi - j0 + 1);
      for (int jj = 0; jj < cnt; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const T* vr = v + (j0 + jj) * kstride + koff;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] = fmaf(pj, to_f32<T>(vr[lane + 32 * c]), acc[c]);
      }
      m = m_new;
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < C; ++c) o[i * qstride + qoff + lane + 32 * c] = from_f32<T>(acc[c] * inv);
    if (lane == 0) lse[((size_t)b * sh.Hq + hq) * sh.sl + i] = m + logf(l);
    __syncwarp();
  }
}

// D_i = sum_d dO_id O_id, one warp per row. D is [bs][Hq][sl] per rank.
template <typename T, int HS>
__global__ void __launch_bounds__(kWarps * 32) attn_bwd_dot_kernel(AttnShape sh, RankPtrs op, RankPtrs dop,
                                                                   float* D) {
  constexpr int C = HS / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.z;
  const int b = blockIdx.y / sh.Hq, hq = blockIdx.y % sh.Hq;
  const T* o = reinterpret_cast<const T*>(op.p[r]);
  const T* dO = reinterpret_cast<const T*>(dop.p[r]);
  const size_t qstride = (size_t)sh.bs * sh.Hq * HS;
  const size_t qoff = ((size_t)b * sh.Hq + hq) * HS;
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int i = blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp + rr;
    if (i >= sh.sl) break;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const size_t e = i * qstride + qoff + lane + 32 * c;
      acc = fmaf(to_f32<T>(o[e]), to_f32<T>(dO[e]), acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) D[(((size_t)r * sh.bs + b) * sh.Hq + hq) * sh.sl + i] = acc;
  }
}

// dQ_i = scale * sum_j P_ij (dO_i . v_j - D_i) k_j, one warp per query row.
template <typename T, int HS>
__global__ void __launch_bounds__(kWarps * 32) attn_bwd_dq_simt_kernel(AttnShape sh, RankPtrs qp, RankPtrs kp,
                                                                       RankPtrs vp, RankPtrs dop, RankPtrs lp,
                                                                       const float* D, RankPtrsMut dqp) {
  constexpr int C = HS / 32;
  __shared__ float qs[kWarps][HS];
  __shared__ float ds_[kWarps][HS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.z;
  const int b = blockIdx.y / sh.Hq, hq = blockIdx.y % sh.Hq, hk = hq / sh.group;
  const T* q = reinterpret_cast<const T*>(qp.p[r]);
  const T* k = reinterpret_cast<const T*>(kp.p[r]);
  const T* v = reinterpret_cast<const T*>(vp.p[r]);
  const T* dO = reinterpret_cast<const T*>(dop.p[r]);
  const float* lse = reinterpret_cast<const float*>(lp.p[r]);
  T* dq = reinterpret_cast<T*>(dqp.p[r]);
  const size_t qstride = (size_t)sh.bs * sh.Hq * HS;
  const size_t kstride = (size_t)sh.bs * sh.Hk * HS;
  const size_t qoff = ((size_t)b * sh.Hq + hq) * HS;
  const size_t koff = ((size_t)b * sh.Hk + hk) * HS;
  const size_t row_base = ((size_t)b * sh.Hq + hq) * sh.sl;
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int i = blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp + rr;
    if (i >= sh.sl) break;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      qs[warp][lane + 32 * c] = to_f32<T>(q[i * qstride + qoff + lane + 32 * c]);
      ds_[warp][lane + 32 * c] = to_f32<T>(dO[i * qstride + qoff + lane + 32 * c]);
    }
    __syncwarp();
    const float L_i = lse[row_base + i];
    const float D_i = D[((size_t)r * sh.bs * sh.Hq) * sh.sl + row_base + i];
    int lo, hi;
    visible_keys(sh, i, lo, hi);
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    for (int j0 = lo; j0 <= hi; j0 += 32) {
      const int j = j0 + lane;
      float dsv = 0.f;
      if (j <= hi) {
        const float s = sh.scale * dot_row<T, HS>(qs[warp], k + j * kstride + koff);
        const float p = expf(s - L_i);
        const float dp = dot_row<T, HS>(ds_[warp], v + j * kstride + koff);
        dsv = p * (dp - D_i);
      }
      const int cnt = min(32, hi - j0 + 1);
      for (int jj = 0; jj < cnt; ++jj) {
        const float d = __shfl_sync(0xffffffffu, dsv, jj);
        const T* kr = k + (j0 + jj) * kstride + koff;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] = fmaf(d, to_f32<T>(kr[lane + 32 * c]), acc[c]);
      }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) dq[i * qstride + qoff + lane + 32 * c] = from_f32<T>(sh.scale * acc[c]);
    __syncwarp();
  }
}

// dV_j = sum_{group} sum_i P_ij dO_i;  dK_j = scale * sum_{group} sum_i dS_ij q_i.
// One warp per key row of one kv head.
template <typename T, int HS>
__global__ void __launch_bounds__(kWarps * 32) attn_bwd_dkdv_simt_kernel(AttnShape sh, RankPtrs qp, RankPtrs kp,
                                                                         RankPtrs vp, RankPtrs dop,
                                                                         RankPtrs lp, const float* D,
                                                                         RankPtrsMut dkp, RankPtrsMut dvp) {
  constexpr int C = HS / 32;
  __shared__ float ks[kWarps][HS];
  __shared__ float vs[kWarps][HS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.z;
  const int b = blockIdx.y / sh.Hk, hk = blockIdx.y % sh.Hk;
  const T* q = reinterpret_cast<const T*>(qp.p[r]);
  const T* k = reinterpret_cast<const T*>(kp.p[r]);
  const T* v = reinterpret_cast<const T*>(vp.p[r]);
  const T* dO = reinterpret_cast<const T*>(dop.p[r]);
  const float* lse = reinterpret_cast<const float*>(lp.p[r]);
  T* dk = reinterpret_cast<T*>(dkp.p[r]);
  T* dv = reinterpret_cast<T*>(dvp.p[r]);
  const size_t qstride = (size_t)sh.bs * sh.Hq * HS;
  const size_t kstride = (size_t)sh.bs * sh.Hk * HS;
  const size_t koff = ((size_t)b * sh.Hk + hk) * HS;
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int j = blockIdx.x * kRowsPerBlock + warp * kRowsPerWarp + rr;
    if (j >= sh.sl) break;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      ks[warp][lane + 32 * c] = to_f32<T>(k[j * kstride + koff + lane + 32 * c]);
      vs[warp][lane + 32 * c] = to_f32<T>(v[j * kstride + koff + lane + 32 * c]);
    }
    __syncwarp();
    int lo, hi;
    visible_queries(sh, j, lo, hi);
    float adk[C], adv[C];
#pragma unroll
    for (int c = 0; c < C; ++c) adk[c] = adv[c] = 0.f;
    for (int gi = 0; gi < sh.group; ++gi) {
      const int hq = hk * sh.group + gi;
      const size_t qoff = ((size_t)b * sh.Hq + hq) * HS;
      const size_t row_base = ((size_t)b * sh.Hq + hq) * sh.sl;
      const float* Dr = D + ((size_t)r * sh.bs * sh.Hq) * sh.sl + row_base;
      for (int i0 = lo; i0 <= hi; i0 += 32) {
        const int i = i0 + lane;
        float p = 0.f, dsv = 0.f;
        if (i <= hi) {
          const float s = sh.scale * dot_row<T, HS>(ks[warp], q + i * qstride + qoff);
          p = expf(s - lse[row_base + i]);
          const float dp = dot_row<T, HS>(vs[warp], dO + i * qstride + qoff);
          dsv = p * (dp - Dr[i]);
        }
        const int cnt = min(32, hi - i0 + 1);
        for (int ii = 0; ii < cnt; ++ii) {
          const float pi = __shfl_sync(0xffffffffu, p, ii);
          const float di = __shfl_sync(0xffffffffu, dsv, ii);
          const T* dor = dO + (i0 + ii) * qstride + qoff;
          const T* qr = q + (i0 + ii) * qstride + qoff;
#pragma unroll
          for (int c = 0; c < C; ++c) {
            adv[c] = fmaf(pi, to_f32<T>(dor[lane + 32 * c]), adv[c]);
            adk[c] = fmaf(di, to_f32<T>(qr[lane + 32 * c]), adk[c]);
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
      dk[j * kstride + koff + lane + 32 * c] = from_f32<T>(sh.scale * adk[c]);
      dv[j * kstride + koff + lane + 32 * c] = from_f32<T>(adv[c]);
    }
    __syncwarp();
  }
}

template <typename T, int HS>
int fwd_simt(const Layer& L, const void* const* q, const void* const* k, const void* const* v,
             void* const* o, float* const* lse, cudaStream_t s) {
  AttnShape sh = make_shape(L);
  RankPtrs Q, K, V;
  RankPtrsMut O, LS;
  for (int r = 0; r < L.P; ++r) {
    Q.p[r] = q[r];
    K.p[r] = k[r];
    V.p[r] = v[r];
    O.p[r] = o[r];
    LS.p[r] = lse[r];
  }
  dim3 grid((unsigned)((L.sl + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)(L.bs * L.Hq), (unsigned)L.P);
  Timed t(L.timing, ULYSSES_KERNEL_ATTN_FWD, s);
  attn_fwd_simt_kernel<T, HS><<<grid, kWarps * 32, 0, s>>>(sh, Q, K, V, O, LS);
  t.done();
  count_launches(1);
  return cuda_status(cudaGetLastError());
}

template <typename T, int HS>
int bwd_simt(const Layer& L, const void* const* q, const void* const* k, const void* const* v,
             const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
             void* const* dk, void* const* dv, void* workspace, cudaStream_t s) {
  AttnShape sh = make_shape(L);
  RankPtrs Q, K, V, O, DO, LS;
  RankPtrsMut DQ, DK, DV;
  for (int r = 0; r < L.P; ++r) {
    Q.p[r] = q[r];
    K.p[r] = k[r];
    V.p[r] = v[r];
    O.p[r] = o[r];
    DO.p[r] = dO[r];
    LS.p[r] = lse[r];
    DQ.p[r] = dq[r];
    DK.p[r] = dk[r];
    DV.p[r] = dv[r];
  }
  // Workspace: the fp32 rows D, [P][bs][Hq][sl].
  float* D = reinterpret_cast<float*>(workspace);
  const unsigned rows = (unsigned)((L.sl + kRowsPerBlock - 1) / kRowsPerBlock);
  Timed t0(L.timing, ULYSSES_KERNEL_BWD_PREP, s);
  attn_bwd_dot_kernel<T, HS><<<dim3(rows, (unsigned)(L.bs * L.Hq), (unsigned)L.P), kWarps * 32, 0, s>>>(sh, O, DO, D);
  t0.done();
  Timed t1(L.timing, ULYSSES_KERNEL_BWD_DQ, s);
  attn_bwd_dq_simt_kernel<T, HS><<<dim3(rows, (unsigned)(L.bs * L.Hq), (unsigned)L.P), kWarps * 32, 0, s>>>(
      sh, Q, K, V, DO, LS, D, DQ);
  t1.done();
  Timed t2(L.timing, ULYSSES_KERNEL_BWD_DKDV, s);
  attn_bwd_dkdv_simt_kernel<T, HS><<<dim3(rows, (unsigned)(L.bs * L.Hk), (unsigned)L.P), kWarps * 32, 0, s>>>(
      sh, Q, K, V, DO, LS, D, DK, DV);
  t2.done();
  count_launches(3);
  return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_attn_fwd_simt(const Layer& L, const void* const* q, const void* const* k, const void* const* v,
                         void* const* o, float* const* lse, cudaStream_t s) {
  if (L.bs * L.Hq > 65535) return ULYSSES_ERR_UNSUPPORTED;
  if (L.dtype == ULYSSES_FP32) {
    switch (L.hs) {
      case 32: return fwd_simt<float, 32>(L, q, k, v, o, lse, s);
      case 64: return fwd_simt<float, 64>(L, q, k, v, o, lse, s);
      case 128: return fwd_simt<float, 128>(L, q, k, v, o, lse, s);
    }
  } else {
    switch (L.hs) {
      case 32: return fwd_simt<__nv_bfloat16, 32>(L, q, k, v, o, lse, s);
      case 64: return fwd_simt<__nv_bfloat16, 64>(L, q, k, v, o, lse, s);
      case 128: return fwd_simt<__nv_bfloat16, 128>(L, q, k, v, o, lse, s);
    }
  }
  return ULYSSES_ERR_UNSUPPORTED;
}

int launch_attn_bwd_simt(const Layer& L, const void* const* q, const void* const* k, const void* const* v,
                         const void* const* o, const void* const* dO, const float* const* lse,
                         void* const* dq, void* const* dk, void* const* dv, void* workspace, cudaStream_t s) {
  if (L.bs * L.Hq > 65535) return ULYSSES_ERR_UNSUPPORTED;
  if (L.dtype == ULYSSES_FP32) {
    switch (L.hs) {
      case 32: return bwd_simt<float, 32>(L, q, k, v, o, dO, lse, dq, dk, dv, workspace, s);
      case 64: return bwd_simt<float, 64>(L, q, k, v, o, dO, lse, dq, dk, dv, workspace, s);
      case 128: return bwd_simt<float, 128>(L, q, k, v, o, dO, lse, dq, dk, dv, workspace, s);
    }
  } else {
    switch (L.hs) {
      case 32: return bwd_simt<__nv_bfloat16, 32>(L, q, k, v, o, dO, lse, dq, dk, dv, workspace, s);
      case 64: return bwd_simt<__nv_bfloat16, 64>(L, q, k, v, o, dO, lse, dq, dk, dv, workspace, s);
      case 128: return bwd_simt<__nv_bfloat16, 128>(L, q, k, v, o, dO, lse, dq, dk, dv, workspace, s);
    }
  }
  return ULYSSES_ERR_UNSUPPORTED;
}

}  // namespace uly
