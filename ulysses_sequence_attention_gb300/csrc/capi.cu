// capi.cu — the extern "C" boundary: handle life cycle, argument checks, dispatch.
//
// Every check in this file runs on the host before anything is enqueued, so a
// rejected call leaves the device untouched. The divisibility rules come from
// the ALST guide ("DeepSpeed Ulysses 序列并行与 Arctic 长序列训练（ALST）集成指南",
// section 2.1, items (5) and (6)). The HF blog ("Ulysses Sequence Parallelism:
// Training with Million-Token Contexts", section "比较 Ulysses 和 Ring Attention")
// requires num_heads >= sp_size.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <new>

#include "internal.cuh"

namespace uly {

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

AttnShape make_shape(const Layer& L) {
  AttnShape s;
  s.sl = (int)L.sl;
  s.bs = (int)L.bs;
  s.P = L.P;
  s.Hq = L.Hq;
  s.Hk = L.Hk;
  s.group = L.Hq / L.Hk;
  s.hs = L.hs;
  s.causal = L.causal;
  s.ndoc = L.ndoc;
  s.scale = (float)(1.0 / sqrt((double)L.hs));
  s.scale_log2 = (float)(1.4426950408889634 / sqrt((double)L.hs));
  s.doc_offsets = L.d_doc_offsets;
  s.status = L.d_status;
  return s;
}

}  // namespace uly

using uly::Layer;

static int check_ptrs(const void* const* ptrs, int P) {
  if (!ptrs) return ULYSSES_ERR_INVALID_ARG;
  for (int r = 0; r < P; ++r) {
    if (!ptrs[r]) return ULYSSES_ERR_INVALID_ARG;
    if (((uintptr_t)ptrs[r]) & 15u) return ULYSSES_ERR_ALIGNMENT;
  }
  return ULYSSES_OK;
}

// Shape rules that do not depend on the sequence length.
static int check_shape(int64_t sl_cap, int64_t bs, int hc, int hkv, int hs, int P, int causal, int dtype) {
  if (sl_cap < 0 || bs < 0 || hc <= 0 || hkv <= 0 || hs <= 0 || P <= 0) return ULYSSES_ERR_INVALID_ARG;
  if (dtype != ULYSSES_BF16 && dtype != ULYSSES_FP32) return ULYSSES_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ULYSSES_ERR_INVALID_ARG;
  // Divisibility rules of the method.
  if (hc % P != 0) return ULYSSES_ERR_DIVISIBILITY;
  if (hc % hkv != 0) return ULYSSES_ERR_DIVISIBILITY;
  if (hkv % P != 0 && P % hkv != 0) return ULYSSES_ERR_DIVISIBILITY;
  // Limits of this build.
  if (P > ULYSSES_MAX_P) return ULYSSES_ERR_UNSUPPORTED;
  if (hs != 32 && hs != 64 && hs != 128) return ULYSSES_ERR_UNSUPPORTED;
  if (sl_cap > (int64_t(1) << 30) || bs > 65535) return ULYSSES_ERR_UNSUPPORTED;
  const int64_t esize = dtype == ULYSSES_BF16 ? 2 : 4;
  if (sl_cap * bs * (int64_t)hc * hs * esize > (int64_t(1) << 38)) return ULYSSES_ERR_UNSUPPORTED;
  return ULYSSES_OK;
}

// Rules on one sequence: sl % P (ALST guide 2.1 (5): the sequence length
// divisible by sp_size) and the document offsets, at which position ids
// restart (ALST guide 2.2).
static int check_seq(int64_t sl, int64_t cap_sl, int P, const int32_t* offs, int ndoc, int cap_docs) {
  if (sl < 0 || sl > cap_sl) return ULYSSES_ERR_INVALID_ARG;
  if (sl % P != 0) return ULYSSES_ERR_DIVISIBILITY;
  if (offs) {
    if (ndoc < 1 || ndoc > cap_docs || offs[0] != 0 || offs[ndoc] != sl) return ULYSSES_ERR_INVALID_ARG;
    for (int d = 0; d < ndoc; ++d)
      if (offs[d + 1] <= offs[d]) return ULYSSES_ERR_INVALID_ARG;
  } else if (ndoc != 0 && ndoc != 1) {
    return ULYSSES_ERR_INVALID_ARG;
  }
  return ULYSSES_OK;
}

static void set_offsets(Layer& L, int64_t sl, const int32_t* offs, int ndoc) {
  L.sl = sl;
  if (offs) {
    L.ndoc = ndoc;
    L.doc_offsets.assign(offs, offs + ndoc + 1);
  } else {
    L.ndoc = 1;
    L.doc_offsets = {0, (int32_t)sl};
  }
}

// Copies the document offsets and, for the tensor-core path, the pair-tile
// schedules of the current sequence into the handle's device tables, which
// hold the capacity. async: in order on `stream` (the host vectors are
// pageable, so each copy has left them when cudaMemcpyAsync returns).
static cudaError_t upload_seq(Layer& L, cudaStream_t stream, bool async) {
  if (L.empty()) return cudaSuccess;
  auto copy = [&](void* dst, const void* src, size_t bytes) {
    return async ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, stream)
                 : cudaMemcpy(dst, src, bytes, cudaMemcpyHostToDevice);
  };
  cudaError_t e = copy(L.d_doc_offsets, L.doc_offsets.data(), sizeof(int32_t) * (L.ndoc + 1));
  if (e == cudaSuccess && uly::fwd_sm103_supported(L)) {
    std::vector<int2> kvp, qp;
    std::vector<int> kvo, qo;
    uly::plan_pair_tiles(L, kvp, kvo, qp, qo);
    std::vector<int> ds_base;
    L.ds_nblk = uly::plan_ds_blocks(kvp, ds_base);
    if (e == cudaSuccess) e = copy(L.d_ds_base, ds_base.data(), sizeof(int) * ds_base.size());
    if (e == cudaSuccess) e = copy(L.d_kvp_range, kvp.data(), sizeof(int2) * kvp.size());
    if (e == cudaSuccess) e = copy(L.d_kvp_order, kvo.data(), sizeof(int) * kvo.size());
    if (e == cudaSuccess) e = copy(L.d_qp_range, qp.data(), sizeof(int2) * qp.size());
    if (e == cudaSuccess) e = copy(L.d_qp_order, qo.data(), sizeof(int) * qo.size());
  }
  return e;
}

static void free_layer(Layer* L) {
  uly::destroy_host_pipe(*L);
  cudaFree(L->d_status);
  cudaFree(L->d_doc_offsets);
  cudaFree(L->d_kvp_range);
  cudaFree(L->d_kvp_order);
  cudaFree(L->d_qp_range);
  cudaFree(L->d_qp_order);
  cudaFree(L->d_ds_base);
  delete L;
}

// A handle whose device tables hold sequences up to cap_sl tokens in up to
// cap_docs documents, set to the sequence (sl, offs).
static int create_layer(ulysses_t* out, int64_t sl, int64_t bs, int hc, int hkv, int hs, int P, int causal,
                        const int32_t* offs, int ndoc, int dtype, int64_t cap_sl, int cap_docs) {
  Layer* L = new (std::nothrow) Layer();
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->bs = bs;
  L->hc = hc;
  L->hkv = hkv;
  L->hs = hs;
  L->P = P;
  L->causal = causal;
  L->dtype = dtype;
  L->Hq = hc / P;
  L->Hk = hkv % P == 0 ? hkv / P : 1;
  L->cap_sl = cap_sl;
  L->cap_docs = cap_docs;
  set_offsets(*L, sl, offs, ndoc);
  if (cudaGetDevice(&L->device) != cudaSuccess) {
    delete L;
    return ULYSSES_ERR_CUDA;
  }
  cudaError_t e = cudaMalloc(&L->d_status, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(L->d_status, 0, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMalloc(&L->d_doc_offsets, sizeof(int32_t) * (cap_docs + 1));
  if (e == cudaSuccess && uly::fwd_sm103_supported(*L) && cap_sl > 0 && bs > 0) {
    const size_t n_pair = (size_t)((cap_sl + 255) / 256);
    e = cudaMalloc(&L->d_kvp_range, sizeof(int2) * n_pair);
    if (e == cudaSuccess) e = cudaMalloc(&L->d_kvp_order, sizeof(int) * n_pair);
    if (e == cudaSuccess) e = cudaMalloc(&L->d_qp_range, sizeof(int2) * n_pair);
    if (e == cudaSuccess) e = cudaMalloc(&L->d_qp_order, sizeof(int) * n_pair);
    if (e == cudaSuccess) e = cudaMalloc(&L->d_ds_base, sizeof(int) * n_pair);
  }
  if (e == cudaSuccess) e = upload_seq(*L, 0, false);
  if (e != cudaSuccess) {
    free_layer(L);
    return ULYSSES_ERR_CUDA;
  }
  uly::noalloc_setup();
  *out = reinterpret_cast<ulysses_t>(L);
  return ULYSSES_OK;
}

#define CHECK_PTRS(arr)                                             \
  do {                                                              \
    int _st = check_ptrs((const void* const*)(arr), L->P);          \
    if (_st != ULYSSES_OK) return _st;                              \
  } while (0)

extern "C" {

const char* ulysses_strerror(int status) {
  switch (status) {
    case ULYSSES_OK: return "ok";
    case ULYSSES_ERR_INVALID_ARG: return "invalid argument";
    case ULYSSES_ERR_DIVISIBILITY: return "divisibility rule broken (sl % P, hc % P, hc % hkv, hkv vs P)";
    case ULYSSES_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case ULYSSES_ERR_UNSUPPORTED: return "unsupported configuration";
    case ULYSSES_ERR_CUDA: return "CUDA runtime error";
    case ULYSSES_ERR_TIMEOUT: return "device-side wait timed out";
    case ULYSSES_ERR_TOO_LARGE: return "larger than a fixed limit (built-in backward scratch, or the handle's capacity)";
    default: return "unknown status";
  }
}

int ulysses_create(ulysses_t* out, int64_t sl, int64_t bs, int hc, int hkv, int hs, int P,
                   int causal, const int32_t* doc_offsets, int ndoc, int dtype) {
  if (!out) return ULYSSES_ERR_INVALID_ARG;
  *out = nullptr;
  int st = check_shape(sl, bs, hc, hkv, hs, P, causal, dtype);
  if (st != ULYSSES_OK) return st;
  st = check_seq(sl, sl, P, doc_offsets, ndoc, doc_offsets ? ndoc : 1);
  if (st != ULYSSES_OK) return st;
  return create_layer(out, sl, bs, hc, hkv, hs, P, causal, doc_offsets, ndoc, dtype, sl, doc_offsets ? ndoc : 1);
}

int ulysses_create_varlen(ulysses_t* out, int64_t max_sl, int64_t bs, int hc, int hkv, int hs, int P, int causal,
                          int max_docs, int dtype) {
  if (!out) return ULYSSES_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_docs < 1) return ULYSSES_ERR_INVALID_ARG;
  int st = check_shape(max_sl, bs, hc, hkv, hs, P, causal, dtype);
  if (st != ULYSSES_OK) return st;
  // Starts empty (sl = 0): every call is a no-op until ulysses_set_seq.
  return create_layer(out, 0, bs, hc, hkv, hs, P, causal, nullptr, 0, dtype, max_sl, max_docs);
}

int ulysses_set_seq(ulysses_t h, int64_t sl, const int32_t* doc_offsets, int ndoc, void* stream) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (sl > L->cap_sl) return ULYSSES_ERR_TOO_LARGE;
  int st = check_seq(sl, L->cap_sl, L->P, doc_offsets, ndoc, L->cap_docs);
  if (st != ULYSSES_OK) return st;
  set_offsets(*L, sl, doc_offsets, ndoc);
  return uly::cuda_status(upload_seq(*L, (cudaStream_t)stream, true));
}

void ulysses_destroy(ulysses_t h) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return;
  free_layer(L);
}

int ulysses_workspace_size(ulysses_t h, size_t* bytes) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L || !bytes) return ULYSSES_ERR_INVALID_ARG;
  *bytes = uly::workspace_bytes(*L, true);
  return ULYSSES_OK;
}

int ulysses_set_ds_budget(ulysses_t h, size_t bytes) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  // As many blocks per (rank, batch, head) as the budget holds, and no more
  // than one document at capacity needs.
  const int64_t cap = uly::ds_blocks_at_capacity(*L);
  const size_t zero = uly::bwd_ds_bytes(*L, 0), per = uly::bwd_ds_bytes(*L, 1) - zero;
  const int64_t fit = bytes > zero ? (int64_t)std::min<size_t>((bytes - zero) / per, (size_t)cap) : 0;
  L->ds_reserved = cap > 0 ? fit : 0;
  return ULYSSES_OK;
}

int ulysses_ds_bytes(ulysses_t h, size_t* needed, size_t* reserved) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  const bool tc = uly::ds_blocks_at_capacity(*L) > 0;
  if (needed) *needed = tc && L->ds_nblk > 0 ? uly::bwd_ds_bytes(*L, L->ds_nblk) : 0;
  if (reserved) *reserved = L->ds_reserved > 0 ? uly::bwd_ds_bytes(*L, L->ds_reserved) : 0;
  return ULYSSES_OK;
}

int ulysses_seq_to_head(ulysses_t h, int nheads, const void* const* seq_shards,
                        void* const* head_shards, void* stream) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (nheads != L->hc && nheads != L->hkv) return ULYSSES_ERR_INVALID_ARG;
  if (L->empty()) return ULYSSES_OK;
  CHECK_PTRS(seq_shards);
  CHECK_PTRS(head_shards);
  return uly::launch_seq_to_head(*L, nheads, seq_shards, head_shards, (cudaStream_t)stream);
}

int ulysses_head_to_seq(ulysses_t h, int nheads, const void* const* head_shards,
                        void* const* seq_shards, void* stream) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (nheads != L->hc && nheads != L->hkv) return ULYSSES_ERR_INVALID_ARG;
  if (L->empty()) return ULYSSES_OK;
  CHECK_PTRS(head_shards);
  CHECK_PTRS(seq_shards);
  return uly::launch_head_to_seq(*L, nheads, head_shards, seq_shards, (cudaStream_t)stream);
}

int ulysses_seq_to_head_qkv(ulysses_t h, const void* const* q_seq, const void* const* k_seq,
                            const void* const* v_seq, void* const* q_head, void* const* k_head, void* const* v_head,
                            void* stream) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (L->empty()) return ULYSSES_OK;
  CHECK_PTRS(q_seq);
  CHECK_PTRS(k_seq);
  CHECK_PTRS(v_seq);
  CHECK_PTRS(q_head);
  CHECK_PTRS(k_head);
  CHECK_PTRS(v_head);
  const int nheads[3] = {L->hc, L->hkv, L->hkv};
  const void* const* src[3] = {q_seq, k_seq, v_seq};
  void* const* dst[3] = {q_head, k_head, v_head};
  return uly::launch_seq_to_head_multi(*L, 3, nheads, src, dst, (cudaStream_t)stream);
}

int ulysses_head_to_seq_qkv(ulysses_t h, const void* const* q_head, const void* const* k_head,
                            const void* const* v_head, void* const* q_seq, void* const* k_seq, void* const* v_seq,
                            void* stream) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (L->empty()) return ULYSSES_OK;
  CHECK_PTRS(q_head);
  CHECK_PTRS(k_head);
  CHECK_PTRS(v_head);
  CHECK_PTRS(q_seq);
  CHECK_PTRS(k_seq);
  CHECK_PTRS(v_seq);
  const int nheads[3] = {L->hc, L->hkv, L->hkv};
  const void* const* src[3] = {q_head, k_head, v_head};
  void* const* dst[3] = {q_seq, k_seq, v_seq};
  return uly::launch_head_to_seq_multi(*L, 3, nheads, src, dst, (cudaStream_t)stream);
}

int ulysses_attn_fwd(ulysses_t h, const void* const* q, const void* const* k,
                     const void* const* v, void* const* o, float* const* lse, void* stream) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (L->empty()) return ULYSSES_OK;
  CHECK_PTRS(q);
  CHECK_PTRS(k);
  CHECK_PTRS(v);
  CHECK_PTRS(o);
  CHECK_PTRS(lse);
  if (uly::fwd_sm103_supported(*L))
    return uly::launch_attn_fwd_sm103(*L, q, k, v, o, lse, (cudaStream_t)stream);
  return uly::launch_attn_fwd_simt(*L, q, k, v, o, lse, (cudaStream_t)stream);
}

int ulysses_attn_bwd(ulysses_t h, const void* const* q, const void* const* k,
                     const void* const* v, const void* const* o, const void* const* dO,
                     const float* const* lse, void* const* dq, void* const* dk, void* const* dv,
                     void* workspace, void* stream) {
  return uly::attn_bwd_entry(h, q, k, v, o, dO, lse, dq, dk, dv, workspace, stream, true);
}

}  // extern "C"

namespace uly {

size_t workspace_bytes(const Layer& L, bool with_ds) {
  // Tensor-core path: per rank two fp32 row planes, -LSE*log2(e) and
  // D = rowsum(dO * O), [bs][Hq][sl rounded up to 4] each, then (stored dS)
  // the zero block and the dS blocks. Other paths: D only, [P][bs][Hq][sl].
  // Sized for the handle's capacity (its own sl unless made by
  // ulysses_create_varlen), so one workspace serves every ulysses_set_seq.
  Layer cap;
  cap.sl = L.cap_sl;
  cap.bs = L.bs;
  cap.P = L.P;
  cap.Hq = L.Hq;
  cap.hs = L.hs;
  cap.dtype = L.dtype;
  if (!fwd_sm103_supported(cap)) return (size_t)cap.P * cap.bs * cap.Hq * cap.sl * sizeof(float);
  if (!with_ds || L.ds_reserved <= 0) return bwd_sm103_workspace(cap);
  return bwd_ds_offset(L) + bwd_ds_bytes(L, L.ds_reserved);
}

// Stored-dS blocks per (rank, batch, head) of the longest sequence the handle
// takes: one document of cap_sl tokens (documents only narrow the ranges).
// 0 when the tensor-core path does not apply or the count leaves int range.
int64_t ds_blocks_at_capacity(const Layer& L) {
  if (!fwd_sm103_supported(L) || L.cap_sl <= 0 || L.bs <= 0) return 0;
  Layer cap;
  cap.sl = L.cap_sl;
  cap.causal = L.causal;
  cap.doc_offsets = {0, (int32_t)L.cap_sl};
  std::vector<int2> kvp, qp;
  std::vector<int> kvo, qo, base;
  plan_pair_tiles(cap, kvp, kvo, qp, qo);
  const int64_t n = plan_ds_blocks(kvp, base);
  return n < 0x7fffffffLL ? n : 0;
}

int attn_bwd_entry(ulysses_t h, const void* const* q, const void* const* k, const void* const* v,
                   const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
                   void* const* dk, void* const* dv, void* workspace, void* stream, bool store_ds) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (L->empty()) return ULYSSES_OK;
  CHECK_PTRS(q);
  CHECK_PTRS(k);
  CHECK_PTRS(v);
  CHECK_PTRS(o);
  CHECK_PTRS(dO);
  CHECK_PTRS(lse);
  CHECK_PTRS(dq);
  CHECK_PTRS(dk);
  CHECK_PTRS(dv);
  if (!workspace) return ULYSSES_ERR_INVALID_ARG;
  if (((uintptr_t)workspace) & 15u) return ULYSSES_ERR_ALIGNMENT;
  if (fwd_sm103_supported(*L))
    return launch_attn_bwd_sm103(*L, q, k, v, o, dO, lse, dq, dk, dv, workspace, (cudaStream_t)stream, false,
                                 store_ds);
  return launch_attn_bwd_simt(*L, q, k, v, o, dO, lse, dq, dk, dv, workspace, (cudaStream_t)stream);
}

}  // namespace uly

extern "C" {

int ulysses_fused_supported(ulysses_t h) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  return uly::fused_supported(*L) ? ULYSSES_OK : ULYSSES_ERR_UNSUPPORTED;
}

int ulysses_layer_fwd(ulysses_t h, const void* const* q, const void* const* k, const void* const* v,
                      void* const* o, float* const* lse, void* stream) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (L->empty()) return ULYSSES_OK;
  if (!uly::fused_supported(*L)) return ULYSSES_ERR_UNSUPPORTED;
  CHECK_PTRS(q);
  CHECK_PTRS(k);
  CHECK_PTRS(v);
  CHECK_PTRS(o);
  CHECK_PTRS(lse);
  return uly::launch_attn_fwd_sm103(*L, q, k, v, o, lse, (cudaStream_t)stream, true);
}

int ulysses_layer_bwd(ulysses_t h, const void* const* q, const void* const* k, const void* const* v,
                      const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
                      void* const* dk, void* const* dv, void* workspace, void* stream) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  L->last_stream = (cudaStream_t)stream;
  if (L->empty()) return ULYSSES_OK;
  if (!uly::fused_supported(*L)) return ULYSSES_ERR_UNSUPPORTED;
  CHECK_PTRS(q);
  CHECK_PTRS(k);
  CHECK_PTRS(v);
  CHECK_PTRS(o);
  CHECK_PTRS(dO);
  CHECK_PTRS(lse);
  CHECK_PTRS(dq);
  CHECK_PTRS(dk);
  CHECK_PTRS(dv);
  if (!workspace) return ULYSSES_ERR_INVALID_ARG;
  if (((uintptr_t)workspace) & 15u) return ULYSSES_ERR_ALIGNMENT;
  return uly::launch_attn_bwd_sm103(*L, q, k, v, o, dO, lse, dq, dk, dv, workspace, (cudaStream_t)stream, true,
                                    true);
}

int ulysses_set_wait_limit(ulysses_t h, int64_t cycles) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L || cycles <= 0) return ULYSSES_ERR_INVALID_ARG;
  L->timeout_cycles = cycles;
  return ULYSSES_OK;
}

int ulysses_inject_fault(ulysses_t h, int kind) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L || kind < 0 || kind > 2) return ULYSSES_ERR_INVALID_ARG;
  L->inject_fault = kind;
  return ULYSSES_OK;
}

uint64_t ulysses_launch_count(void) { return uly::g_launches.load(std::memory_order_relaxed); }

int ulysses_timing_enable(ulysses_t h, int enable) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  if (enable) L->timing.reset();
  L->timing.on = enable != 0;
  return L->timing.failed ? ULYSSES_ERR_CUDA : ULYSSES_OK;
}

int ulysses_timing_read(ulysses_t h, int kernel, double* total_ms, int64_t* launches) {
  Layer* L = reinterpret_cast<Layer*>(h);
  if (!L || kernel < 0 || kernel >= ULYSSES_KERNEL_COUNT) return ULYSSES_ERR_INVALID_ARG;
  L->timing.drain(L->timing.pending.size());
  if (total_ms) *total_ms = L->timing.total_ms[kernel];
  if (launches) *launches = L->timing.launches[kernel];
  return L->timing.failed ? ULYSSES_ERR_CUDA : ULYSSES_OK;
}

int ulysses_get_status(ulysses_t h) {
  const Layer* L = reinterpret_cast<const Layer*>(h);
  if (!L) return ULYSSES_ERR_INVALID_ARG;
  // In order on the stream of the handle's latest call: the read follows that
  // stream's work, the clear precedes anything enqueued on it later, and only
  // that stream is waited for.
  const cudaStream_t s = L->last_stream;
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, L->d_status, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ULYSSES_ERR_CUDA;
  if (cudaMemsetAsync(L->d_status, 0, sizeof(unsigned), s) != cudaSuccess) return ULYSSES_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ULYSSES_ERR_CUDA;
  if (word & uly::STATUS_TIMEOUT) return ULYSSES_ERR_TIMEOUT;
  return ULYSSES_OK;
}

}  // extern "C"
