/*
 * ulysses.h — C ABI of the GB300 Ulysses sequence-parallel attention layer.
 *
 * The layer is DeepSpeed-Ulysses as the pages describe it. The HF blog
 * "Ulysses Sequence Parallelism: Training with Million-Token Contexts" lists
 * the algorithm steps: sequence sharding, QKV projection, all-to-all, local
 * attention, all-to-all, output projection. The DeepSpeed-Ulysses blog
 * ("DeepSpeed Ulysses: 训练极长序列Transformer模型的系统优化", section
 * "DeepSpeed-Ulysses的核心设计") gives the core design. This library is the
 * path between the projections:
 *
 *   P sequence shards [sl/P, bs, H, hs]
 *     --seq->head exchange-->  P head shards [sl, bs, H/P, hs]
 *     --exact causal softmax attention, forward and backward, per head-->
 *     --head->seq exchange-->  P sequence shards [sl/P, bs, H, hs]
 *
 * All P ranks are shard buffers on ONE GPU. An exchange is a permutation
 * from HBM to HBM, not a collective between GPUs.
 *
 * Conventions shared by every call:
 *  - Layout. Sequence-major HF layout: a sequence shard is [sl/P][bs][H][hs]
 *    and a head shard is [sl][bs][H/P][hs], row-major (hs fastest). The source
 *    is the ALST guide ("DeepSpeed Ulysses 序列并行与 Arctic 长序列训练（ALST）集成指南",
 *    section 1, which fixes the shape [sl, bs, hc, hs]). Rank i holds tokens
 *    [i*sl/P, (i+1)*sl/P). After seq->head it holds heads [r*H/P, (r+1)*H/P).
 *    This is the 2-GPU diagram of the Transformers guide, section
 *    "Ulysses 序列并行的核心原理".
 *  - GQA. Query head h reads kv head h / (hc/hkv). When P > hkv, rank r holds
 *    kv head r*hkv/P (replication, ALST guide section 2.1 item (6)).
 *  - Pointers. Every tensor argument is a HOST array of P DEVICE pointers,
 *    one per virtual rank. Each pointer must be non-NULL and 16-byte aligned.
 *    The caller owns every device buffer, including the workspace, and keeps
 *    it alive until the work queued on the stream has finished.
 *  - Streams. `stream` is a cudaStream_t (NULL = legacy default stream). Every
 *    device call only enqueues work on it and returns without synchronising.
 *    The one exception is ulysses_get_status, which waits for one stream.
 *  - Errors. Every int-returning call returns ULYSSES_OK (0) or a negative
 *    ulysses_status. No C++ exception crosses this boundary. Arguments are
 *    checked before anything is enqueued. A failed check enqueues nothing.
 *  - Element types. ULYSSES_BF16 (bfloat16) or ULYSSES_FP32 for
 *    Q/K/V/O/dO/dQ/dK/dV. The logsumexp is always fp32. Exchanges copy bits;
 *    they never convert.
 */
#ifndef ULYSSES_H
#define ULYSSES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque handle. It owns only small metadata (shape, a device copy of the
 * document offsets, a device status word). Created by ulysses_create, freed by
 * ulysses_destroy. A handle may be used from one host thread at a time. */
typedef struct ulysses_layer* ulysses_t;

typedef enum ulysses_status {
  ULYSSES_OK = 0,
  ULYSSES_ERR_INVALID_ARG = -1,  /* NULL pointer, bad dtype, malformed document offsets, bad nheads */
  ULYSSES_ERR_DIVISIBILITY = -2, /* one of the pages' divisibility rules is broken (see ulysses_create) */
  ULYSSES_ERR_ALIGNMENT = -3,    /* a device pointer is not 16-byte aligned */
  ULYSSES_ERR_UNSUPPORTED = -4,  /* valid for the method, but outside what this build implements */
  ULYSSES_ERR_CUDA = -5,         /* a CUDA runtime call failed (allocation, launch) */
  ULYSSES_ERR_TIMEOUT = -6,      /* a device-side bounded wait ran out (reported by ulysses_get_status) */
  ULYSSES_ERR_TOO_LARGE = -7     /* beyond a fixed size: the scratch of ulysses_attn_bwd_noalloc, the capacity of ulysses_set_seq */
} ulysses_status;

typedef enum ulysses_dtype {
  ULYSSES_BF16 = 0,
  ULYSSES_FP32 = 1
} ulysses_dtype;

#define ULYSSES_MAX_P 128

/*
 * ulysses_create — validate a layer shape and build a handle.
 *
 *   sl      global sequence length (all P shards together). 0 is allowed:
 *           the handle then describes an empty layer and every call is a no-op.
 *   bs      batch size (0 allowed, as for sl).
 *   hc      query heads; hkv key/value heads; hs head size (32, 64 or 128).
 *   P       sequence-parallel degree (virtual ranks), 1 <= P <= ULYSSES_MAX_P.
 *           P = 1 is legal: the exchanges become plain copies.
 *   causal  1: key j is visible from query i only when j <= i; 0: all keys
 *           of the same document are visible.
 *   doc_offsets  HOST array of ndoc+1 int32 document start offsets in the
 *           global sequence: [0] = 0, strictly increasing, [ndoc] = sl. Or NULL
 *           for one document. Position ids restart at each offset, so no key
 *           is visible across a document boundary. This is the packed-sequence
 *           rule of the ALST guide, section 2.2. The handle keeps its own copy.
 *   dtype   ulysses_dtype of the activation tensors.
 *
 * Divisibility (ULYSSES_ERR_DIVISIBILITY; ALST guide section 2.1 items (5)
 * and (6); HF blog section "比较 Ulysses 和 Ring Attention", which requires
 * num_heads >= sp_size):
 *   sl % P == 0;  hc % P == 0 (so P <= hc);  hc % hkv == 0;
 *   hkv % P == 0 or P % hkv == 0.
 * On any error *out is set to NULL. Allocates a few bytes of device memory on
 * the current device.
 */
int ulysses_create(ulysses_t* out, int64_t sl, int64_t bs, int hc, int hkv, int hs, int P,
                   int causal, const int32_t* doc_offsets, int ndoc, int dtype);

/*
 * ulysses_create_varlen — a handle for batches of varying sequence length:
 * the pages' `seq_length_is_variable=True` mode (ALST guide, section 2.1 item
 * (5); HF blog, the DeepSpeedSequenceParallelConfig options). ulysses_create is
 * the fixed mode (`seq_length_is_variable=False`), whose shapes are computed
 * once.
 *
 *   max_sl    the longest sequence the handle will take (capacity).
 *   max_docs  the most documents a sequence may be packed from (>= 1).
 *   others    as for ulysses_create; the same shape and divisibility rules,
 *             except that sl % P is checked per sequence by ulysses_set_seq.
 * The handle starts empty (sl = 0): every call is a no-op until the first
 * ulysses_set_seq. Its device tables are sized for the capacity, and
 * ulysses_workspace_size reports the workspace for max_sl, so one set of
 * buffers serves every sequence. Allocates a few bytes of device memory per
 * 256 tokens of capacity on the current device.
 */
int ulysses_create_varlen(ulysses_t* out, int64_t max_sl, int64_t bs, int hc, int hkv, int hs, int P,
                          int causal, int max_docs, int dtype);

/*
 * ulysses_set_seq — switch a handle to a new sequence: length and document
 * offsets. Works on any handle within its capacity (ulysses_create's capacity
 * is its own sl and document count).
 *
 *   sl           new global sequence length, 0 <= sl <= capacity, sl % P == 0
 *                (ULYSSES_ERR_DIVISIBILITY otherwise; ULYSSES_ERR_TOO_LARGE
 *                above the capacity). 0 makes every call a no-op.
 *   doc_offsets  HOST array of ndoc+1 offsets as for ulysses_create, with
 *                ndoc <= max_docs; or NULL (one document).
 *   stream       the new tile schedule and offsets are copied to the device in
 *                order on this stream. Calls enqueued after this one on the same
 *                stream use the new sequence; work of this handle already
 *                enqueued on other streams must be finished or ordered before
 *                `stream`. The host arrays may be freed on return.
 * Buffers passed to later calls take the new sl: a sequence shard is
 * [sl/P][bs][H][hs], a head shard [sl][bs][H/P][hs], LSE [bs][hc/P][sl].
 * Allocates nothing. A failed check changes nothing and enqueues nothing.
 */
int ulysses_set_seq(ulysses_t h, int64_t sl, const int32_t* doc_offsets, int ndoc, void* stream);

/* Free the handle and its device metadata. NULL is a no-op. The caller must
 * make sure that no work using the handle is still running. */
void ulysses_destroy(ulysses_t h);

/* Static text for a status code. Never NULL. */
const char* ulysses_strerror(int status);

/*
 * ulysses_workspace_size — bytes of device workspace that ulysses_attn_bwd needs,
 * at the handle's capacity (its sl; max_sl for ulysses_create_varlen).
 * bf16 with hs = 128 (the tensor-core path): for each rank, two fp32 row
 * planes [bs][hc/P][pitch], -LSE*log2(e) and D = rowsum(dO * O), where pitch
 * is sl rounded up to a multiple of 4: P * 2 * bs * (hc/P) * pitch * 4 bytes.
 * Other configurations: D only, P * bs * (hc/P) * sl * 4 bytes. With a dS
 * area reserved (ulysses_set_ds_budget), add it after the row planes, at an
 * offset rounded up to 1024 bytes (`reserved` of ulysses_ds_bytes). Pure
 * host computation.
 */
int ulysses_workspace_size(ulysses_t h, size_t* bytes);

/*
 * ulysses_set_ds_budget — reserve up to `bytes` of the workspace for keeping
 * dS (default 0: none).
 *
 * dQ_i = s * sum_j dS_ij k_j needs the same dS_ij = P_ij (dO_i . v_j - D_i)
 * that the dK/dV pass forms (HF blog "Ulysses Sequence Parallelism", the
 * per-head backward of algorithm step 4; the attention backward it runs is
 * the flash-attention one). With stored dS on, the dK/dV kernel also writes
 * the bf16 dS of every 128 x 128 block of visible (query, key) pairs, and dQ
 * becomes one GEMM per block that reads it back, instead of recomputing S
 * and dP (two more GEMMs and the exponentials). It costs 2 bytes per visible
 * pair and head: for a causal sequence of sl tokens, about
 * bs * hc * sl^2 bytes (34.6 GB for sl = 32768, bs = 1, hc = 32); packed
 * documents need only their own pairs.
 *
 *   bytes  the budget. The area reserved is a 32 KB zero block plus as many
 *          64 KB blocks per (rank, batch, query head) as fit in `bytes`, but
 *          no more than one document of the handle's capacity needs (the
 *          most any of its sequences can). Nothing is reserved below the
 *          zero block and one block, or off the tensor-core path (bf16,
 *          hs = 128).
 * A backward stores dS when the blocks of the current sequence fit the
 * reserved area (ulysses_ds_bytes: needed <= reserved), and recomputes dQ
 * otherwise; ulysses_attn_bwd_noalloc always recomputes. Changes
 * ulysses_workspace_size: query it again after this call and pass a
 * workspace of that size to every later ulysses_attn_bwd / ulysses_layer_bwd.
 * dK and dV are unchanged bit for bit; dQ agrees with the recomputing path
 * within bf16 rounding (its dS is formed by the other kernel). Pure host
 * computation. ULYSSES_ERR_INVALID_ARG for a NULL handle.
 */
int ulysses_set_ds_budget(ulysses_t h, size_t bytes);

/*
 * ulysses_ds_bytes — stored-dS sizes, in bytes (either pointer may be NULL):
 *   needed    the area the current sequence uses: a 32 KB zero block, then
 *             per (rank, batch, query head) 64 KB per visible pair of
 *             (256-key tile, 128-query tile); 0 off the tensor-core path or
 *             for an empty sequence.
 *   reserved  the area reserved in the workspace (ulysses_set_ds_budget), 0
 *             if none.
 * Pure host computation. ULYSSES_ERR_INVALID_ARG for a NULL handle.
 */
int ulysses_ds_bytes(ulysses_t h, size_t* needed, size_t* reserved);

/*
 * ulysses_seq_to_head — the first all-to-all: re-shard from sequence to heads.
 * HF blog algorithm step 3. Transformers guide: the first all-to-all moves the
 * sharded dimension from the sequence to the heads.
 *
 *   nheads       hc (for Q or dO) or hkv (for K or V).
 *   seq_shards   P device pointers, each [sl/P][bs][nheads][hs] (input).
 *   head_shards  P device pointers, each [sl][bs][nheads/P][hs] (output). When
 *                P > nheads, each is [sl][bs][1][hs] with head r*nheads/P.
 *   head_shards[r][t][b][j][:] = seq_shards[t/(sl/P)][t%(sl/P)][b][r*nheads/P + j][:]
 * A bit-exact copy. Input and output buffers must not overlap.
 */
int ulysses_seq_to_head(ulysses_t h, int nheads, const void* const* seq_shards,
                        void* const* head_shards, void* stream);

/*
 * ulysses_head_to_seq — the second all-to-all: back from heads to sequence.
 * HF blog algorithm step 5. DeepSpeed-Ulysses blog, section
 * "DeepSpeed-Ulysses的核心设计": after attention, a second all-to-all turns
 * the output back into the N/P sequence layout.
 *
 *   nheads       hc (O, dQ) or hkv (dK, dV).
 *   head_shards  P device pointers, each [sl][bs][nheads/P][hs] (input).
 *   seq_shards   P device pointers, each [sl/P][bs][nheads][hs] (output).
 * A bit-exact copy when nheads % P == 0. When P > nheads (replicated kv heads),
 * the input is a gradient. The output for head h is then the sum of the
 * P/nheads replicas. The sum runs in fp32 and is rounded once to the element
 * type.
 */
int ulysses_head_to_seq(ulysses_t h, int nheads, const void* const* head_shards,
                        void* const* seq_shards, void* stream);

/*
 * ulysses_seq_to_head_qkv — the layer's first all-to-all for Q, K and V
 * together, in one launch: the 3Nh message of the DeepSpeed-Ulysses blog,
 * section "显著的通信量减少". Each tensor is exchanged exactly as
 * ulysses_seq_to_head would (Q with hc heads, K and V with hkv heads, with kv
 * replication when P > hkv). One launch covers all three, so the K and V
 * exchanges, too small to fill the GPU on their own, share the Q
 * exchange's waves.
 *   q_seq, k_seq, v_seq     P sequence shards each (inputs)
 *   q_head, k_head, v_head  P head shards each (outputs)
 */
int ulysses_seq_to_head_qkv(ulysses_t h, const void* const* q_seq, const void* const* k_seq,
                            const void* const* v_seq, void* const* q_head, void* const* k_head,
                            void* const* v_head, void* stream);

/*
 * ulysses_head_to_seq_qkv — the backward's last all-to-all for dQ, dK and dV
 * together: ulysses_head_to_seq of each (dQ with hc heads, dK and dV with
 * hkv heads), in one launch. When P > hkv the replica sums of dK and dV need
 * their own kernel, and the three exchanges then run as three launches.
 *   q_head, k_head, v_head  P head shards each (inputs: dQ, dK, dV)
 *   q_seq, k_seq, v_seq     P sequence shards each (outputs)
 */
int ulysses_head_to_seq_qkv(ulysses_t h, const void* const* q_head, const void* const* k_head,
                            const void* const* v_head, void* const* q_seq, void* const* k_seq,
                            void* const* v_seq, void* stream);

/*
 * ulysses_attn_fwd — local exact attention of every rank's head group.
 * HF blog algorithm step 4 (standard attention per head; heads are
 * independent). The DeepSpeed-Ulysses blog's per-head equation did not survive
 * extraction. The equation implemented is the SDPA/FlashAttention definition:
 *
 *   S_ij = q_i . k_j / sqrt(hs)
 *   O_i  = sum_j softmax_j(S_ij over visible j) v_j
 *   LSE_i = ln sum_{visible j} exp(S_ij)
 *
 *   q, o     P pointers, each [sl][bs][hc/P][hs] (head shards)
 *   k, v     P pointers, each [sl][bs][Hk][hs], Hk = max(hkv/P, 1)
 *   lse      P pointers, each fp32 [bs][hc/P][sl] (output, kept for backward)
 * Softmax and the accumulation run in fp32. O is rounded once to the element
 * type (round to nearest even for bf16).
 */
int ulysses_attn_fwd(ulysses_t h, const void* const* q, const void* const* k,
                     const void* const* v, void* const* o, float* const* lse, void* stream);

/*
 * ulysses_attn_bwd — gradients of the local attention for L with dL/dO = dO.
 * The backward of the layer is the reverse of the forward: dO goes through
 * seq->head, this call runs, and dQ/dK/dV go through head->seq.
 *
 *   D_i   = sum_d dO_id O_id
 *   P_ij  = exp(S_ij - LSE_i)       (visible j; 0 otherwise)
 *   dV_j  = sum_{q heads of the group} sum_i P_ij dO_i
 *   dS_ij = P_ij (dO_i . v_j - D_i)
 *   dQ_i  = sum_j dS_ij k_j / sqrt(hs)
 *   dK_j  = sum_{q heads of the group} sum_i dS_ij q_i / sqrt(hs)
 *
 *   q, o, dO, dq   [sl][bs][hc/P][hs] per rank; k, v, dk, dv [sl][bs][Hk][hs]
 *   lse            the forward's fp32 [bs][hc/P][sl] per rank
 *   workspace      device buffer of ulysses_workspace_size bytes, 16-byte
 *                  aligned, owned by the caller. Its contents on entry are
 *                  ignored and on exit are unspecified.
 */
int ulysses_attn_bwd(ulysses_t h, const void* const* q, const void* const* k,
                     const void* const* v, const void* const* o, const void* const* dO,
                     const float* const* lse, void* const* dq, void* const* dk, void* const* dv,
                     void* workspace, void* stream);

/*
 * ulysses_layer_fwd — the whole forward of the layer in one call: the
 * seq->head exchange of Q, K and V, the local attention of ulysses_attn_fwd,
 * and the head->seq exchange of O. HF blog algorithm steps 3 to 5. The
 * DeepSpeed-Ulysses blog, section "DeepSpeed-Ulysses的核心设计", places local
 * attention between the two all-to-alls.
 *
 * On one GPU the exchange is a permutation of addresses. Here it is fused
 * into the attention kernel: its TMA loads read each tile straight from the
 * sequence shard that holds those tokens, and its epilogue stores O straight
 * into the sequence shard of its rows. No head-shard copy is made, and no
 * exchange kernel runs. The results are bit-identical to ulysses_seq_to_head +
 * ulysses_attn_fwd + ulysses_head_to_seq.
 *
 *   q, o     P pointers, each [sl/P][bs][hc][hs]  (sequence shards)
 *   k, v     P pointers, each [sl/P][bs][hkv][hs] (sequence shards)
 *   lse      P pointers, each fp32 [bs][hc/P][sl] (output, head layout as in
 *            ulysses_attn_fwd: rank r's heads [r*hc/P, (r+1)*hc/P))
 * Returns ULYSSES_ERR_UNSUPPORTED, and enqueues nothing, unless
 * ulysses_fused_supported(h) is ULYSSES_OK. The explicit three-call path
 * covers every other shape.
 */
int ulysses_layer_fwd(ulysses_t h, const void* const* q, const void* const* k, const void* const* v,
                      void* const* o, float* const* lse, void* stream);

/*
 * ulysses_layer_bwd — the whole backward of the layer in one call: dO
 * seq->head, ulysses_attn_bwd, and dQ, dK, dV head->seq, with both exchanges
 * fused into the kernels' TMA addressing as in ulysses_layer_fwd.
 *
 *   q, o, dO, dq   P pointers, each [sl/P][bs][hc][hs]  (sequence shards)
 *   k, v, dk, dv   P pointers, each [sl/P][bs][hkv][hs] (sequence shards)
 *   lse            the forward's fp32 [bs][hc/P][sl] per rank
 *   workspace      ulysses_workspace_size bytes, as for ulysses_attn_bwd
 * Bit-identical to the explicit path. ULYSSES_ERR_UNSUPPORTED (nothing
 * enqueued) unless ulysses_fused_supported(h) is ULYSSES_OK.
 */
int ulysses_layer_bwd(ulysses_t h, const void* const* q, const void* const* k, const void* const* v,
                      const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
                      void* const* dk, void* const* dv, void* workspace, void* stream);

/*
 * ulysses_fused_supported — ULYSSES_OK if ulysses_layer_fwd/_bwd accept this
 * handle, else ULYSSES_ERR_UNSUPPORTED. They need all of:
 *   - dtype ULYSSES_BF16 and hs = 128 (the tensor-core kernels);
 *   - P <= 8 (a launch holds one TMA tensor map per shard and operand);
 *   - sl/P a multiple of 128, so that no 128-row tile spans two shards;
 *   - hkv % P == 0 (replicated kv heads need the replica sum of
 *     ulysses_head_to_seq).
 * An empty layer (sl = 0 or bs = 0) reports what its shape would allow; the
 * layer calls are no-ops for it either way. Host only.
 */
int ulysses_fused_supported(ulysses_t h);

/*
 * Host-streaming training steps: ulysses_host_begin, ulysses_host_step,
 * ulysses_host_end.
 *
 * A step is what a training loop feeds the layer. The P sequence shards of Q,
 * K, V and dO come from HOST memory. The layer runs forward and backward (as
 * ulysses_layer_fwd + ulysses_layer_bwd), and O, dQ, dK, dV go back to host
 * memory. In the pages' loop each rank's DataLoader hands it its sequence
 * shard (ALST guide, section 2.2: the DataLoader adapter and its CPU prefetch
 * buffer). Here the P shards of a step are P host buffers per tensor.
 *
 * The copies run on two copy streams owned by the handle (host->device and
 * device->host). The kernels run on `stream`. With two slots of device
 * buffers, used alternately, step i+1's inputs travel while step i computes,
 * and step i's outputs travel while step i+1 computes. The library orders
 * every reuse of a slot with events:
 *   - the copy of inputs into a slot waits for the last compute on that slot;
 *   - its forward waits for the last copy of outputs out of the slot;
 *   - the copy of O starts when the forward ends and overlaps the backward.
 *
 * ulysses_host_begin(h, stream): the copy streams wait for the work already
 *   enqueued on `stream`. Call it once before a run of steps.
 * ulysses_host_end(h, stream): `stream` waits for every copy enqueued so far.
 *   After it, an event recorded on `stream`, or a synchronisation of `stream`,
 *   covers all the steps' copies and kernels.
 * ulysses_host_step(h, slot, host_in, host_out, dev, lse, workspace, stream):
 *   slot       0 or 1: which set of device buffers `dev` is.
 *   host_in    4*P HOST pointers: Q shards 0..P-1, then K, V and dO. Use
 *              pinned memory: pageable memory works, but the copies then stop
 *              overlapping. Keep them unchanged until ulysses_host_end and a
 *              synchronisation of `stream`.
 *   host_out   4*P HOST pointers: O, dQ, dK, dV. Written asynchronously; valid
 *              after ulysses_host_end and a synchronisation of `stream`.
 *   dev        8*P DEVICE pointers of this slot: Q, K, V, dO, O, dQ, dK, dV,
 *              each [sl/P][bs][H][hs] (H = hc or hkv). They must not be used
 *              elsewhere while the steps run.
 *   lse        P DEVICE pointers, fp32 [bs][hc/P][sl], shared by both slots.
 *   workspace  ulysses_workspace_size bytes of DEVICE memory, shared by both slots.
 *   Every pointer must be non-NULL; device pointers must be 16-byte aligned.
 *   Shapes must be accepted by ulysses_fused_supported (ULYSSES_ERR_UNSUPPORTED
 *   otherwise, with nothing enqueued). The first call of a handle creates its two
 *   copy streams and a few events. It allocates no device memory. Everything
 *   is enqueued; nothing synchronises.
 * There is no counterpart of the streams and slots on the pages: they are how
 * this library keeps the host copies off the critical path.
 */
int ulysses_host_begin(ulysses_t h, void* stream);
int ulysses_host_step(ulysses_t h, int slot, const void* const* host_in, void* const* host_out,
                      void* const* dev, float* const* lse, void* workspace, void* stream);
int ulysses_host_end(ulysses_t h, void* stream);

/*
 * ulysses_get_status — read and clear the handle's device status word.
 * The read and the clear are enqueued on the stream of the handle's latest
 * call that took a stream, and this call waits for that stream only: work of
 * the handle enqueued on other streams must be ordered before it by the
 * caller. Returns ULYSSES_OK, ULYSSES_ERR_TIMEOUT if a bounded device-side
 * wait ran out since the last call (the kernel then returned early and its
 * outputs are invalid), or ULYSSES_ERR_CUDA if the stream reports an error.
 */
int ulysses_get_status(ulysses_t h);

/*
 * ulysses_set_wait_limit — bound, in SM clock cycles, on every device-side
 * wait of the tensor-core kernels (mbarrier waits between warps, TMA and
 * UMMA completions). The default is 4e9 cycles (about 2 s). A wait that
 * runs out sets the handle's status word, and the kernel winds down without
 * touching more data; ulysses_get_status then returns ULYSSES_ERR_TIMEOUT.
 * cycles must be positive (ULYSSES_ERR_INVALID_ARG otherwise). Host only.
 */
int ulysses_set_wait_limit(ulysses_t h, int64_t cycles);

/*
 * ulysses_inject_fault — test hook for the failure path; never needed in use.
 *   kind 0: no fault (clears a pending one).
 *   kind 1: in the next tensor-core forward call, the TMA producer issues no
 *           K/V loads, so the waits for them run out. Combine with a short
 *           ulysses_set_wait_limit. The injection is consumed by that call.
 *   kind 2: the same for the next tensor-core backward call: the dK/dV
 *           kernel's producer issues no Q/dO tile loads. dK and dV are then
 *           invalid; dQ is computed as usual.
 * Nothing faults, traps or hangs: every wait is bounded. Returns
 * ULYSSES_ERR_INVALID_ARG for an unknown kind. Host only.
 */
int ulysses_inject_fault(ulysses_t h, int kind);

/*
 * ulysses_launch_count — number of CUDA kernels this library has enqueued
 * since it was loaded, over all handles and threads. A diagnostic counter for
 * benchmarks: the difference across a region is the number of launches the
 * region made. Never fails.
 */
uint64_t ulysses_launch_count(void);

/* The kernels of the library, as ulysses_timing_read counts them. */
typedef enum ulysses_kernel {
  ULYSSES_KERNEL_SEQ_TO_HEAD = 0,  /* seq->head exchange */
  ULYSSES_KERNEL_HEAD_TO_SEQ = 1,  /* head->seq exchange, with the replica sum if P > nheads */
  ULYSSES_KERNEL_ATTN_FWD = 2,     /* attention forward: O and LSE */
  ULYSSES_KERNEL_BWD_PREP = 3,     /* backward, D = rowsum(dO * O) per query row */
  ULYSSES_KERNEL_BWD_DKDV = 4,     /* backward, dK and dV */
  ULYSSES_KERNEL_BWD_DQ = 5,       /* backward, dQ */
  ULYSSES_KERNEL_COUNT = 6
} ulysses_kernel;

/*
 * ulysses_timing_enable — per-kernel device time of one handle, for
 * benchmarks. There is no counterpart in the paper.
 *
 * enable != 0 clears the handle's totals and starts timing. From then on,
 * every kernel that a call of this handle enqueues is bracketed by two CUDA
 * events recorded on the call's stream, so the time between them is that
 * kernel's device time. enable == 0 stops timing; launches already timed
 * stay readable. The events cost a few microseconds of host time per launch
 * and do not change what the kernels compute. Returns ULYSSES_OK, or
 * ULYSSES_ERR_CUDA if an event could not be created. Host only.
 */
int ulysses_timing_enable(ulysses_t h, int enable);

/*
 * ulysses_timing_read — device time and launch count of one kernel since the
 * last ulysses_timing_enable(h, 1). kernel is a ulysses_kernel. This call
 * waits for the events that the timed launches recorded (it blocks until
 * that work has finished). total_ms and launches are host pointers; each may
 * be NULL. Returns ULYSSES_ERR_INVALID_ARG for an unknown kernel and
 * ULYSSES_ERR_CUDA if an event could not be recorded or read.
 */
int ulysses_timing_read(ulysses_t h, int kernel, double* total_ms, int64_t* launches);

/*
 * ulysses_attn_bwd_noalloc — ulysses_attn_bwd for callers that cannot allocate
 * device memory. There is no counterpart in the paper: this is a deployment
 * convenience of this library.
 *
 * Who needs it: code that runs inside another runtime which owns the GPU's
 * memory. Examples are a plugin that is handed only its input and output
 * buffers, a server that reserves all device memory at start-up and must not
 * allocate while it serves, and a framework whose caching allocator has to
 * account for every byte. Such callers cannot call cudaMalloc for the
 * workspace that ulysses_attn_bwd takes. cudaMalloc can also synchronise the
 * device, which stalls work on other streams.
 *
 * Arguments and results are those of ulysses_attn_bwd, without `workspace`.
 * The workspace is a file-scope device array of
 * ULYSSES_NOALLOC_SCRATCH_BYTES bytes inside the library. Every GPU on which
 * a handle has been created holds this array until the process exits. This
 * call never calls cudaMalloc, cudaFree or any allocating library routine.
 * The handle still comes from ulysses_create, which allocates a few bytes of
 * metadata and sets up the array (below): create it during set-up.
 *
 * Limits and sharing:
 *  - A layer whose backward needs more than ULYSSES_NOALLOC_SCRATCH_BYTES of
 *    workspace (ulysses_workspace_size without the stored-dS area) is
 *    rejected with ULYSSES_ERR_TOO_LARGE before anything is enqueued. The
 *    workspace is 8 bytes per (token, query head, batch element) on the
 *    tensor-core path: 64 MiB covers, for example, 256K tokens of a
 *    32-query-head layer. This call never stores dS (ulysses_set_ds_budget):
 *    dQ is recomputed.
 *  - Every call shares the one array, and it keeps the last call's contents.
 *    Each call clears the parts that must start at zero itself. Two calls that
 *    overlap on the GPU (on different streams, or different host threads
 *    without ordering) race on the array and corrupt each other's gradients:
 *    order them.
 *  - The array's device address comes from cudaGetSymbolAddress, looked up
 *    by ulysses_create (and ulysses_create_varlen) on the current device.
 *    That lookup loads the array on the device: its 64 MiB are committed
 *    when the first handle of a device is created, not when the library is
 *    loaded. A call of this function then allocates nothing. If that lookup
 *    failed, the first call here tries once more and returns
 *    ULYSSES_ERR_CUDA if it fails again; make that call before any stream
 *    capture begins. A cudaDeviceReset destroys the array with every handle
 *    of the device; handles created after it look the array up again.
 */
#define ULYSSES_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int ulysses_attn_bwd_noalloc(ulysses_t h, const void* const* q, const void* const* k,
                             const void* const* v, const void* const* o, const void* const* dO,
                             const float* const* lse, void* const* dq, void* const* dk,
                             void* const* dv, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ULYSSES_H */
