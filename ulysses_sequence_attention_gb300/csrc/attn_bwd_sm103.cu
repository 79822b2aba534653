// attn_bwd_sm103.cu — attention backward on the tcgen05 tensor cores.
//
// The backward of the layer reverses its forward (HF blog "Ulysses Sequence
// Parallelism: Training with Million-Token Contexts", algorithm steps 3-5):
// dO goes seq->head, this runs per head, and dQ/dK/dV go head->seq. Per head,
// with s = 1/sqrt(hs), P_ij = exp(s q_i.k_j - LSE_i) on visible pairs:
//   D_i = dO_i . O_i,  dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - D_i),
//   dQ_i = s sum_j dS_ij k_j,  dK_j = s sum_i dS_ij q_i
// and the kv gradients of a GQA group sum over its query heads.
//
// Three kernels:
//  1. bwd_prep: D = rowsum(dO * O) in fp32, and the fp32 dQ accumulator set to zero.
//  2. bwd_main: one CTA per (rank, batch, kv head, 128-key tile). It keeps K and
//     V in shared memory and loops over every query head of the group and every
//     128-row query tile that can see the keys (causal and per-document block
//     skipping). Per query tile the tensor core computes
//        S^T = K Q^T,  dP^T = V dO^T                      (into tensor memory)
//        dV += P^T dO,  dK += dS^T Q                      (accumulated in tensor memory)
//        dQ_tile = dS K                                   (into tensor memory)
//     and eight compute warps turn S^T, dP^T into P^T and dS^T (bf16) between
//     the two halves. A fourth warpgroup reads each dQ tile out of tensor
//     memory, stages it in the consumed Q/dO stage and adds it into the fp32
//     accumulator with TMA reduce-add (whole 128-byte lines at L2). At the end
//     dK (scaled by s) and dV leave by TMA store.
//  3. bwd_dq_convert: dQ = bf16(accumulator).
//
// Tensor memory: [0,128) S^T, then P^T (bf16) in [0,64); [128,256) dP^T, then
// dS^T (bf16) in [128,192), then the dQ tile; [256,384) dV; [384,512) dK.
// Reuse relies on UMMAs from one thread running in issue order.
//
// Warp roles (512 threads): warps 0-7 compute (thread = kv row / TMEM lane,
// warp w handles columns [64*(w/4), 64*(w/4)+64)); warp 8 TMA and the LSE/D
// rows; warp 9 UMMA and tensor-memory allocation; warps 10-11 complete the
// third warpgroup; warps 12-15 move the dQ tiles. Every mbarrier wait is
// bounded.
#include <math.h>

#include <algorithm>
#include <numeric>
#include <vector>

#include "internal.cuh"
#include "sm103.cuh"
#include "tmap.cuh"

namespace uly {
namespace {
using namespace sm103;

constexpr int kRanksPerLaunch = 8;
constexpr int kThreads = 512;
// Registers: the block launches at 128 per thread; the compute warpgroups take
// 160, the TMA/UMMA warpgroup keeps 56, the dQ warpgroup 136 (a whole dQ row
// in flight): 2*128*160 + 128*56 + 128*136 = 512*128.
constexpr int kRegsLaunch = (65536 / kThreads) / 8 * 8;  // registers per thread at launch
constexpr int kRegsCompute = 160;
constexpr int kRegsIssue = 56;
constexpr int kRegsDq = 136;
// setmaxnreg.inc may only raise and .dec only lower a warpgroup's count, and
// the raises must be paid for by the releases.
static_assert(kRegsCompute >= kRegsLaunch && kRegsDq >= kRegsLaunch && kRegsIssue <= kRegsLaunch,
              "register split directions");
static_assert(2 * 128 * kRegsCompute + 128 * kRegsIssue + 128 * kRegsDq <= kThreads * kRegsLaunch,
              "register split must add up to the launch budget");
constexpr int NQ = 2;                              // Q/dO pipeline stages
constexpr uint32_t kTile = 128 * 128 * 2;          // 32 KB
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kTile;
constexpr uint32_t kOffQ = 2 * kTile;              // NQ tiles
constexpr uint32_t kOffDO = kOffQ + NQ * kTile;    // NQ tiles
constexpr uint32_t kOffDS = kOffDO + NQ * kTile;   // 1 tile
constexpr uint32_t kOffRow = kOffDS + kTile;       // NQ x (128 LSE + 128 D) floats
constexpr uint32_t kOffBar = kOffRow + NQ * 1024;
constexpr uint32_t kSmemBytes = kOffBar + 256;     // the dynamic base must be 1024-aligned

struct BwdParams {
  CUtensorMap tq[kRanksPerLaunch];
  CUtensorMap tk[kRanksPerLaunch];
  CUtensorMap tv[kRanksPerLaunch];
  CUtensorMap tdo[kRanksPerLaunch];
  CUtensorMap tdk[kRanksPerLaunch];
  CUtensorMap tdv[kRanksPerLaunch];
  CUtensorMap tdq[kRanksPerLaunch];    // fp32 accumulator [sl][bs][Hq][128], boxes of 32 x 128
  const float* lse[kRanksPerLaunch];
  const float* D[kRanksPerLaunch];     // [bs][Hq][sl]
  const int2* q_range;                 // per key tile: first and last query tile
  const int* n_order;                  // key tiles, most work first
  const int32_t* doc_offsets;
  unsigned* status;
  long long timeout;
  int ndoc, sl, bs, Hq, Hk, group, nranks, causal;
  float scale, scale_log2;
};

enum {
  B_KVFULL = 0,
  B_QFULL = 1,                 // NQ: Q, dO tiles and their LSE/D rows (32 arrivals + tx)
  B_QEMPTY = B_QFULL + NQ,     // NQ: the stage's dQ reduction has read it (1)
  B_SFULL = B_QEMPTY + NQ,     // S^T done (commit)
  B_DPFULL = B_SFULL + 1,      // dP^T done (commit)
  B_LOADED = B_DPFULL + 1,     // compute warps hold S^T, dP^T in registers (256)
  B_PFULL = B_LOADED + 1,      // P^T, dS^T written (256)
  B_DQFULL = B_PFULL + 1,      // dQ tile done (commit)
  B_DQEMPTY = B_DQFULL + 1,    // dQ tile read out of tensor memory (128)
  B_STAGED = B_DQEMPTY + 1,    // dQ tile staged in shared memory (128)
  B_DKDV = B_STAGED + 1,       // every UMMA done (commit)
  B_EPI = B_DKDV + 1,          // dK/dV staged (256)
  B_DRAIN = B_EPI + 1,
  B_COUNT
};

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_sm103_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // the layout needs a 1024-byte aligned base; report instead of misreading
    if (threadIdx.x == 0) atomicOr(p.status, STATUS_TIMEOUT);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  float* rows = reinterpret_cast<float*>(smem + kOffRow);  // [NQ][2][128]: LSE*log2(e), D

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Work item: (key tile, rank, batch, kv head).
  const int units = p.nranks * p.bs * p.Hk;
  const int n = p.n_order[blockIdx.x / units];
  int rest = blockIdx.x % units;
  const int hk = rest % p.Hk;
  rest /= p.Hk;
  const int b = rest % p.bs;
  const int rl = rest / p.bs;
  const int2 qr = p.q_range[n];
  const int nm = qr.y - qr.x + 1;
  const int n_it = p.group * nm;

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_LOADED || i == B_PFULL || i == B_EPI) cnt = 256;
      if (i == B_DQEMPTY || i == B_STAGED) cnt = 128;
      if (i >= B_QFULL && i < B_QFULL + NQ) cnt = 32;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = p.timeout;

  if (warp >= 8 && warp < 12) {
    regs_dec<kRegsIssue>();
    if (warp == 8) {
      // ------------------------------------------------------------- TMA producer
      bool ok = true;
      int last_q[NQ];
      for (int i = 0; i < NQ; ++i) last_q[i] = -1;
      if (lane == 0) {
        mbar_expect_tx(bar(B_KVFULL), 2 * kTile);
        tma_load_4d(sb + kOffK, &p.tk[rl], bar(B_KVFULL), 0, hk, b, n * 128);
        tma_load_4d(sb + kOffK + kTile / 2, &p.tk[rl], bar(B_KVFULL), 64, hk, b, n * 128);
        tma_load_4d(sb + kOffV, &p.tv[rl], bar(B_KVFULL), 0, hk, b, n * 128);
        tma_load_4d(sb + kOffV + kTile / 2, &p.tv[rl], bar(B_KVFULL), 64, hk, b, n * 128);
      }
      for (int it = 0; it < n_it; ++it) {
        const int st = it % NQ, u = it / NQ;
        const int hq = hk * p.group + it / nm;
        const int m = qr.x + it % nm;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B_QEMPTY + st), (u & 1) ^ 1, lim));
        if (!ok) break;
        // LSE (in log2 units) and D of the tile's 128 rows; rows past the end
        // get LSE = +inf, so that P = 0 there.
        float* rs = rows + st * 256;
        const size_t base = ((size_t)b * p.Hq + hq) * p.sl;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = m * 128 + lane * 4 + e;
          const bool in = i < p.sl;
          rs[lane * 4 + e] = in ? p.lse[rl][base + i] * 1.4426950408889634f : INFINITY;
          rs[128 + lane * 4 + e] = in ? p.D[rl][base + i] : 0.f;
        }
        if (lane == 0) {
          mbar_expect_tx(bar(B_QFULL + st), 2 * kTile);
          const uint32_t dq = sb + kOffQ + st * kTile, ddo = sb + kOffDO + st * kTile;
          tma_load_4d(dq, &p.tq[rl], bar(B_QFULL + st), 0, hq, b, m * 128);
          tma_load_4d(dq + kTile / 2, &p.tq[rl], bar(B_QFULL + st), 64, hq, b, m * 128);
          tma_load_4d(ddo, &p.tdo[rl], bar(B_QFULL + st), 0, hq, b, m * 128);
          tma_load_4d(ddo + kTile / 2, &p.tdo[rl], bar(B_QFULL + st), 64, hq, b, m * 128);
        } else {
          mbar_arrive(bar(B_QFULL + st));
        }
        last_q[st] = u;
      }
      if (lane == 0) {
        if (!ok) atomicOr(p.status, STATUS_TIMEOUT);
        mbar_wait(bar(B_KVFULL), 0, lim);
        for (int i = 0; i < NQ; ++i)
          if (last_q[i] >= 0) mbar_wait(bar(B_QFULL + i), last_q[i] & 1, lim);
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------- UMMA issuer
      // Per query tile i, in issue order:
      //   dV += P_i^T dO_i and dK += dS_i^T Q_i, interleaved (two independent
      //   accumulators keep the tensor pipe fed);
      //   S_{i+1}^T = K Q_{i+1}^T                     (commit: S ready)
      //   dQ_i = dS_i K                               (commit: dQ ready)
      //   dP_{i+1}^T = V dO_{i+1}^T, once dQ_i is read out  (commit: dP ready)
      // so the exponentials of tile i+1 overlap dQ_i and its readout.
      if (lane == 0) {
        constexpr uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);   // K-major x K-major
        constexpr uint32_t id_tm = idesc_bf16_f32(128, 128, 0, 1);   // tmem A x MN-major B
        constexpr uint32_t id_mm = idesc_bf16_f32(128, 128, 1, 1);   // MN-major A x MN-major B
        const uint32_t sK = sb + kOffK, sV = sb + kOffV, sDS = sb + kOffDS;
        auto kmaj = [](uint32_t base, int kk) {
          return sdesc_sw128(base + (kk >> 2) * (kTile / 2) + (kk & 3) * 32, 0, 1024);
        };
        auto mnmaj = [](uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, kTile / 2, 1024); };
        auto issue_s = [&](int st) {
          const uint32_t sQ = sb + kOffQ + st * kTile;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) umma_ss(tmem + 0, kmaj(sK, kk), kmaj(sQ, kk), id_kk, kk > 0);
        };
        auto issue_dp = [&](int st) {
          const uint32_t sDO = sb + kOffDO + st * kTile;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) umma_ss(tmem + 128, kmaj(sV, kk), kmaj(sDO, kk), id_kk, kk > 0);
        };
        bool ok = mbar_wait(bar(B_KVFULL), 0, lim) && mbar_wait(bar(B_QFULL), 0, lim);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          umma_commit(bar(B_SFULL));
          issue_dp(0);
          umma_commit(bar(B_DPFULL));
        }
        for (int it = 0; it < n_it && ok; ++it) {
          const int st = it % NQ;
          const bool next = it + 1 < n_it;
          const int st1 = (it + 1) % NQ, u1 = (it + 1) / NQ;
          const uint32_t sQ = sb + kOffQ + st * kTile, sDO = sb + kOffDO + st * kTile;
          if (!mbar_wait(bar(B_PFULL), it & 1, lim)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dV += P^T dO and dK += dS^T Q
            const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
            umma_ts(tmem + 256, tmem + 0 + kk * 8, mnmaj(sDO, kk), id_tm, acc);
            umma_ts(tmem + 384, tmem + 128 + kk * 8, mnmaj(sQ, kk), id_tm, acc);
          }
          if (next) {
            if (!mbar_wait(bar(B_QFULL + st1), u1 & 1, lim)) { ok = false; break; }
            tc_fence_after();
            issue_s(st1);
            umma_commit(bar(B_SFULL));
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ tile = dS K
            umma_ss(tmem + 128, mnmaj(sDS, kk), mnmaj(sK, kk), id_mm, kk > 0);
          umma_commit(bar(B_DQFULL));
          if (next) {
            if (!mbar_wait(bar(B_DQEMPTY), it & 1, lim)) { ok = false; break; }
            tc_fence_after();
            issue_dp(st1);
            umma_commit(bar(B_DPFULL));
          }
        }
        if (ok)
          umma_commit(bar(B_DKDV));
        else
          atomicOr(p.status, STATUS_TIMEOUT);
        umma_commit(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, lim);
      }
      __syncwarp();
    }
  } else if (warp >= 12) {
    regs_inc<kRegsDq>();
    // --------------------------------------------------------------- dQ warpgroup
    // Row qi of the dQ tile (TMEM lane) goes, scaled by s, into the consumed
    // Q/dO stage as four 128x32 fp32 boxes (128-byte swizzled); one thread
    // then adds them into the fp32 accumulator with TMA reduce-add.
    const int quarter = warp & 3;
    const int rq = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % NQ;
      const int m = qr.x + it % nm;
      const int hq = hk * p.group + it / nm;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_DQFULL), it & 1, lim));
      if (!ok) break;
      tc_fence_after();
      uint32_t g[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tmem + lane_base + 128 + 32 * q, g[q]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(B_DQEMPTY));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // box q: columns [32q, 32q+32); Q stage holds boxes 0-1, dO stage boxes 2-3
        const uint32_t box = (q < 2 ? sb + kOffQ + st * kTile : sb + kOffDO + st * kTile) + (q & 1) * (kTile / 2);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = box + sw128_offset(rq, c);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                       "f"(p.scale * __uint_as_float(g[q][4 * c])), "f"(p.scale * __uint_as_float(g[q][4 * c + 1])),
                       "f"(p.scale * __uint_as_float(g[q][4 * c + 2])), "f"(p.scale * __uint_as_float(g[q][4 * c + 3]))
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_STAGED));
      if (rq == 0) {
        if (mbar_wait(bar(B_STAGED), it & 1, lim)) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t box = (q < 2 ? sb + kOffQ + st * kTile : sb + kOffDO + st * kTile) + (q & 1) * (kTile / 2);
            tma_reduce_add_4d(&p.tdq[rl], box, 32 * q, hq, b, m * 128);
          }
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(bar(B_QEMPTY + st));
        } else {
          ok = false;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
    }
    if (rq == 0) bulk_wait_all();
    if (!ok && lane == 0) atomicOr(p.status, STATUS_TIMEOUT);
  } else {
    regs_inc<kRegsCompute>();
    // --------------------------------------------------------------- compute warps
    const int quarter = warp & 3;
    const int h = warp >> 2;                   // column half
    const int jr = quarter * 32 + lane;        // kv row within the tile = TMEM lane
    const int j = n * 128 + jr;                // global key position
    int qlo = 1, qhi = 0;                      // queries that see key j: [qlo, qhi]
    if (j < p.sl) {
      const int d = doc_of(p.doc_offsets, p.ndoc, j);
      qlo = p.causal ? j : p.doc_offsets[d];
      qhi = p.doc_offsets[d + 1] - 1;
    }
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % NQ;
      const int m = qr.x + it % nm;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_SFULL), it & 1, lim) &&
                                       mbar_wait(bar(B_QFULL + st), (it / NQ) & 1, lim));
      if (!ok) break;
      tc_fence_after();
      uint32_t pf[64];
      tmem_ld32(tmem + lane_base + 0 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pf[0]));
      tmem_ld32(tmem + lane_base + 32 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pf[32]));
      tmem_ld_wait();
      const float* rs = rows + st * 256;
      const int i0 = m * 128 + 64 * h;           // first query of this thread's columns
      const bool full = qlo <= i0 && i0 + 63 <= qhi;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float pv = ex2_approx(fmaf(__uint_as_float(pf[c]), sl2, -rs[64 * h + c]));
        if (!full) {
          const int i = i0 + c;
          if (i < qlo || i > qhi) pv = 0.f;
        }
        pf[c] = __float_as_uint(pv);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_DPFULL), it & 1, lim));
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[64];
      tmem_ld32(tmem + lane_base + 128 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tmem + lane_base + 160 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_ld_wait();
      // Both column halves must be read before either half is overwritten.
      tc_fence_before();
      mbar_arrive(bar(B_LOADED));
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = __uint_as_float(pf[2 * c]), p1 = __uint_as_float(pf[2 * c + 1]);
        const float d0 = p0 * (__uint_as_float(dp[2 * c]) - rs[128 + 64 * h + 2 * c]);
        const float d1 = p1 * (__uint_as_float(dp[2 * c + 1]) - rs[128 + 64 * h + 2 * c + 1]);
        pk[c] = pack_bf16x2(p0, p1);
        dk[c] = pack_bf16x2(d0, d1);
      }
      // dS^T row jr, queries [64h, 64h+64): one 128-byte row of half h of the
      // swizzled smem tile (the MN-major A operand of dQ = dS K). The previous
      // dQ UMMA finished before dP^T of this tile was committed.
      const uint32_t ds_row = sb + kOffDS + h * (kTile / 2);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = ds_row + sw128_offset(jr, c);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(dk[4 * c]), "r"(dk[4 * c + 1]),
                     "r"(dk[4 * c + 2]), "r"(dk[4 * c + 3])
                     : "memory");
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(B_LOADED), it & 1, lim));
      if (!ok) break;
      tc_fence_after();
      tmem_st32(tmem + lane_base + 0 + 32 * h, pk);      // P^T, bf16
      tmem_st32(tmem + lane_base + 128 + 32 * h, dk);    // dS^T, bf16
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(B_DKDV), 0, lim));
    if (ok) {
      tc_fence_after();
      // dV (cols 256+) and dK (cols 384+, times s) of kv row jr, columns [64h,64h+64),
      // staged into the V and K tiles (free now) and stored by TMA.
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t col = (which == 0 ? 256 : 384) + 64 * h;
        const uint32_t stage = sb + (which == 0 ? kOffV : kOffK) + h * (kTile / 2);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + col + 32 * q, o);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[c4 * 8 + 2 * e]) * mul, __uint_as_float(o[c4 * 8 + 2 * e + 1]) * mul);
            const uint32_t addr = stage + sw128_offset(jr, q * 4 + c4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_EPI));
      if (threadIdx.x == 0) {
        if (mbar_wait(bar(B_EPI), 0, lim)) {
          tma_store_4d(&p.tdv[rl], sb + kOffV, 0, hk, b, n * 128);
          tma_store_4d(&p.tdv[rl], sb + kOffV + kTile / 2, 64, hk, b, n * 128);
          tma_store_4d(&p.tdk[rl], sb + kOffK, 0, hk, b, n * 128);
          tma_store_4d(&p.tdk[rl], sb + kOffK + kTile / 2, 64, hk, b, n * 128);
          bulk_commit();
          bulk_wait_all();
        } else {
          atomicOr(p.status, STATUS_TIMEOUT);
        }
      }
    } else if (lane == 0) {
      atomicOr(p.status, STATUS_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D = rowsum(dO * O) for every (rank, batch, head, row), and dq_acc = 0.
// Eight lanes per row, 16 bytes of O and of dO per lane.
struct PrepParams {
  const __nv_bfloat16* o[ULYSSES_MAX_P];
  const __nv_bfloat16* dO[ULYSSES_MAX_P];
  float* D[ULYSSES_MAX_P];
  float4* dq_acc[ULYSSES_MAX_P];
  int P, sl, bs, Hq;
  long long rows_per_rank;      // sl * bs * Hq
  long long acc_vec_per_rank;   // sl * bs * Hq * 32
};

__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const __grid_constant__ PrepParams a) {
  const long long total_rows = a.rows_per_rank * a.P;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  // 16 threads per row: 8 bf16 of O and of dO each. The loop runs whole
  // warps (the shuffle below needs every lane); lanes past the end add zeros.
  const long long lane = threadIdx.x & 31;
  for (long long g = tid; g - lane < total_rows * 16; g += nthreads) {
    const bool active = g < total_rows * 16;
    const long long row = active ? (g >> 4) : 0;
    const int part = (int)(g & 15);
    const int r = (int)(row / a.rows_per_rank);
    const long long rr = row - (long long)r * a.rows_per_rank;  // (t, b, hq)
    float acc = 0.f;
    if (active) {
      const uint4 ov = *reinterpret_cast<const uint4*>(a.o[r] + rr * 128 + part * 8);
      const uint4 dv = *reinterpret_cast<const uint4*>(a.dO[r] + rr * 128 + part * 8);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(o2[e]);
        const float2 df = __bfloat1622float2(d2[e]);
        acc = fmaf(of.x, df.x, fmaf(of.y, df.y, acc));
      }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (active && part == 0) {
      const int hq = (int)(rr % a.Hq);
      const long long tb = rr / a.Hq;
      const int bb = (int)(tb % a.bs);
      const long long t = tb / a.bs;
      a.D[r][((long long)bb * a.Hq + hq) * a.sl + t] = acc;
    }
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long g = tid; g < a.acc_vec_per_rank * a.P; g += nthreads) {
    const int r = (int)(g / a.acc_vec_per_rank);
    a.dq_acc[r][g - (long long)r * a.acc_vec_per_rank] = z;
  }
}

struct ConvParams {
  const float4* acc[ULYSSES_MAX_P];
  __nv_bfloat16* dq[ULYSSES_MAX_P];
  int P;
  long long vec_per_rank;
};

__global__ void __launch_bounds__(256) attn_bwd_dq_convert_kernel(const __grid_constant__ ConvParams a) {
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < a.vec_per_rank * a.P; g += nthreads) {
    const int r = (int)(g / a.vec_per_rank);
    const long long e = g - (long long)r * a.vec_per_rank;
    const float4 v = a.acc[r][e];
    uint2 out;
    out.x = pack_bf16x2(v.x, v.y);
    out.y = pack_bf16x2(v.z, v.w);
    reinterpret_cast<uint2*>(a.dq[r])[e] = out;
  }
}

}  // namespace

void plan_bwd_tiles(const Layer& L, std::vector<int2>& q_range, std::vector<int>& order) {
  const int sl = (int)L.sl;
  const int n_n = (sl + 127) / 128;
  q_range.resize(n_n);
  std::vector<int> cost(n_n);
  auto doc = [&](int t) {
    return (int)(std::upper_bound(L.doc_offsets.begin(), L.doc_offsets.end(), t) - L.doc_offsets.begin()) - 1;
  };
  for (int n = 0; n < n_n; ++n) {
    const int first = n * 128, last = std::min(sl, first + 128) - 1;
    const int lo_q = L.causal ? first : L.doc_offsets[doc(first)];
    const int hi_q = L.doc_offsets[doc(last) + 1] - 1;
    q_range[n] = make_int2(lo_q / 128, hi_q / 128);
    cost[n] = q_range[n].y - q_range[n].x + 1;
  }
  order.resize(n_n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int c) { return cost[a] > cost[c]; });
}

static int grid_cap(long long work) {
  long long g = (work + 255) / 256;
  return (int)std::max(1LL, std::min(g, 152LL * 16));
}

int launch_attn_bwd_sm103(const Layer& L, const void* const* q, const void* const* k, const void* const* v,
                          const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
                          void* const* dk, void* const* dv, void* workspace, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_bwd_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
      return ULYSSES_ERR_CUDA;
    attr_set = true;
  }
  const long long per_rank_acc = (long long)L.sl * L.bs * L.Hq * L.hs;  // floats
  float* acc_base = reinterpret_cast<float*>(workspace);
  float* D_base = acc_base + per_rank_acc * L.P;
  const long long per_rank_D = (long long)L.bs * L.Hq * L.sl;

  // 1. D and zeroed accumulators.
  {
    PrepParams a;
    for (int r = 0; r < L.P; ++r) {
      a.o[r] = reinterpret_cast<const __nv_bfloat16*>(o[r]);
      a.dO[r] = reinterpret_cast<const __nv_bfloat16*>(dO[r]);
      a.D[r] = D_base + per_rank_D * r;
      a.dq_acc[r] = reinterpret_cast<float4*>(acc_base + per_rank_acc * r);
    }
    a.P = L.P;
    a.sl = (int)L.sl;
    a.bs = (int)L.bs;
    a.Hq = L.Hq;
    a.rows_per_rank = (long long)L.sl * L.bs * L.Hq;
    a.acc_vec_per_rank = per_rank_acc / 4;
    attn_bwd_prep_kernel<<<grid_cap(a.rows_per_rank * L.P * 16), 256, 0, stream>>>(a);
    count_launches(1);
  }
  // 2. Main kernel, in launches of up to kRanksPerLaunch ranks.
  BwdParams prm;
  prm.q_range = L.d_q_range;
  prm.n_order = L.d_n_order;
  prm.doc_offsets = L.d_doc_offsets;
  prm.status = L.d_status;
  prm.timeout = L.timeout_cycles;
  prm.ndoc = L.ndoc;
  prm.sl = (int)L.sl;
  prm.bs = (int)L.bs;
  prm.Hq = L.Hq;
  prm.Hk = L.Hk;
  prm.group = L.Hq / L.Hk;
  prm.causal = L.causal;
  prm.scale = (float)(1.0 / sqrt((double)L.hs));
  prm.scale_log2 = (float)(1.4426950408889634 / sqrt((double)L.hs));
  const int n_n = (int)((L.sl + 127) / 128);
  for (int r0 = 0; r0 < L.P; r0 += kRanksPerLaunch) {
    const int nr = std::min(kRanksPerLaunch, L.P - r0);
    prm.nranks = nr;
    for (int i = 0; i < nr; ++i) {
      const int r = r0 + i;
      bool ok = make_tmap_bf16_4d(&prm.tq[i], q[r], 128, L.Hq, L.bs, L.sl, 64, 128) &&
                make_tmap_bf16_4d(&prm.tk[i], k[r], 128, L.Hk, L.bs, L.sl, 64, 128) &&
                make_tmap_bf16_4d(&prm.tv[i], v[r], 128, L.Hk, L.bs, L.sl, 64, 128) &&
                make_tmap_bf16_4d(&prm.tdo[i], dO[r], 128, L.Hq, L.bs, L.sl, 64, 128) &&
                make_tmap_bf16_4d(&prm.tdk[i], dk[r], 128, L.Hk, L.bs, L.sl, 64, 128) &&
                make_tmap_bf16_4d(&prm.tdv[i], dv[r], 128, L.Hk, L.bs, L.sl, 64, 128);
      if (!ok) return ULYSSES_ERR_CUDA;
      if (!make_tmap_f32_4d(&prm.tdq[i], acc_base + per_rank_acc * r, 128, L.Hq, L.bs, L.sl, 32, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B))
        return ULYSSES_ERR_CUDA;
      prm.lse[i] = lse[r];
      prm.D[i] = D_base + per_rank_D * r;
    }
    const long long grid = (long long)n_n * nr * L.bs * L.Hk;
    if (grid > 0x7fffffffLL) return ULYSSES_ERR_UNSUPPORTED;
    attn_bwd_sm103_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(prm);
    count_launches(1);
  }
  // 3. dQ to bf16.
  {
    ConvParams a;
    for (int r = 0; r < L.P; ++r) {
      a.acc[r] = reinterpret_cast<const float4*>(acc_base + per_rank_acc * r);
      a.dq[r] = reinterpret_cast<__nv_bfloat16*>(dq[r]);
    }
    a.P = L.P;
    a.vec_per_rank = per_rank_acc / 4;
    attn_bwd_dq_convert_kernel<<<grid_cap(a.vec_per_rank * L.P), 256, 0, stream>>>(a);
    count_launches(1);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace uly
