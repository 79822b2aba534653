// attn_bwd_sm103.cu — attention backward on the tcgen05 tensor cores, two SMs per tile.
//
// The backward of the layer reverses its forward (HF blog "Ulysses Sequence
// Parallelism: Training with Million-Token Contexts", algorithm steps 3-5):
// dO goes seq->head, this runs per head, and dQ/dK/dV go head->seq. Per head,
// with s = 1/sqrt(hs), P_ij = exp(s q_i.k_j - LSE_i) on visible pairs:
//   D_i = dO_i . O_i,  dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - D_i),
//   dQ_i = s sum_j dS_ij k_j,  dK_j = s sum_i dS_ij q_i
// and the kv gradients of a GQA group sum over its query heads.
//
// Three kernels, no atomics:
//  1. bwd_prep: D = rowsum(dO * O) in fp32.
//  2. bwd_dkdv: a CTA pair owns 256 keys (128 per CTA) of one kv head. For every
//     query head of the group and every 128-row query tile that can see the keys
//     (causal and per-document block skipping), the pair computes with M = 256
//     UMMAs (tcgen05 .cta_group::2, issued by the even CTA):
//        S^T = K Q^T,  dP^T = V dO^T                 (tensor memory)
//        dV += P^T dO,  dK += dS^T Q                 (accumulated in tensor memory)
//     and eight compute warps per CTA turn S^T, dP^T into P^T, dS^T (bf16),
//     both written over dP^T, so that S^T of the next tile can be issued
//     while dV and dK of this one still run. At the end dK (times s) and dV
//     leave by TMA store.
//  3. bwd_dq: a CTA pair owns 256 queries of one query head and loops over the
//     visible key tiles:
//        S = Q K^T,  dP = dO V^T,  dQ += dS K        (M = 256 UMMAs)
//     with dS written in place over dP as the tensor-memory A operand.
// Recomputing S and dP for dQ costs two more GEMMs per tile than accumulating
// dQ with atomics, but M = 256 UMMAs run at about twice the rate of the M = 128
// form, and dQ needs no fp32 reduction traffic.
//
// In a pair, the B operand of each UMMA is split along N: for N = queries (or
// keys) each CTA holds 64 of the 128 rows; for N = head dimension each CTA
// holds 64 of its 128 columns. TMA loads of the odd CTA complete on its own
// barriers and are forwarded to the even CTA's barriers with a remote arrive.
// Every mbarrier wait is bounded.
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
constexpr int kThreads = 384;
constexpr int kRegsLaunch = (65536 / kThreads) / 8 * 8;  // registers per thread at launch
constexpr int kRegsCompute = 224;
constexpr int kRegsOther = 56;
static_assert(kRegsCompute >= kRegsLaunch && kRegsOther <= kRegsLaunch, "register split directions");
static_assert(2 * 128 * kRegsCompute + 128 * kRegsOther <= kThreads * kRegsLaunch,
              "register split must add up to the launch budget");
constexpr uint32_t kTile = 128 * 128 * 2;  // a 128x128 bf16 tile: 32 KB
constexpr uint32_t kHalf = kTile / 2;      // 16 KB

static_assert(kMaxFusedP <= kRanksPerLaunch, "a fused launch holds one tensor map per sequence shard");

// Tensor maps ta..th: one per rank of the launch (head shards), or one per
// sequence shard (fused; see locate_tile). tr and rows are per rank.
struct PairParams {
  CUtensorMap ta[kRanksPerLaunch];   // dkdv: K 64x128     dq: Q 64x128
  CUtensorMap tb[kRanksPerLaunch];   // dkdv: V 64x128     dq: dO 64x128
  CUtensorMap tc[kRanksPerLaunch];   // dkdv: Q 64x64      dq: K 64x64
  CUtensorMap td[kRanksPerLaunch];   // dkdv: dO 64x64     dq: V 64x64
  CUtensorMap te[kRanksPerLaunch];   // dkdv: Q 64x128     dq: K 64x128
  CUtensorMap tf[kRanksPerLaunch];   // dkdv: dO 64x128    dq: dQ (store)
  CUtensorMap tg[kRanksPerLaunch];   // dkdv: dK (store)
  CUtensorMap th[kRanksPerLaunch];   // dkdv: dV (store)
  CUtensorMap tr[kRanksPerLaunch];   // dkdv: the row planes (-LSE log2 e, D) of a rank, boxes of 128 x 1 x 2
  const float* rows[kRanksPerLaunch];  // dq: the row planes of a rank, [2][bs*Hq][pitch]
  const int2* range;                 // per pair tile: first and last tile of the other side
  const int* order;                  // pair tiles, most work first
  char* ds;                          // dkdv: stored dS blocks of the launch's first rank, or null
  const int* ds_base;                // dkdv: first block of each key pair tile in a (rank, batch, head)
  long long ds_nblk;                 // dkdv: blocks per (rank, batch, head)
  const int32_t* doc_offsets;
  unsigned* status;
  long long timeout;
  int ndoc, sl, bs, Hq, Hk, group, nranks, causal;
  int fused;                         // operands are sequence shards of n tokens (nranks = P)
  int n;
  int pitch;                         // floats per row of a row plane (sl rounded up to 4)
  int skip_q_loads;                  // test hook (dK/dV): the producer issues no Q/dO tile loads
  float scale, scale_log2;
};

__device__ __forceinline__ void pair_status(const PairParams& p) { atomicOr(p.status, STATUS_TIMEOUT); }

// Stage a thread's row of a 128-row x 64-column bf16 block (64 values as 32
// packed words), 128-byte swizzled, at `region`.
__device__ __forceinline__ void stage_row64(uint32_t region, int row, const uint32_t (&w)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t addr = region + sw128_offset(row, c);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[4 * c]), "r"(w[4 * c + 1]),
                 "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                 : "memory");
  }
}

// ===========================================================================
// dK / dV: pair = 256 keys
// ===========================================================================
namespace dkdv {
constexpr int NQ = 2;
constexpr uint32_t kOffK = 0, kOffV = kTile;
// Per stage: Qn, dOn (this CTA's 64 query rows x 128, K-major), then Qh, dOh
// (all 128 query rows x this CTA's 64 head columns, MN-major).
constexpr uint32_t kOffStage = 2 * kTile;
constexpr uint32_t kStage = 4 * kHalf;
constexpr uint32_t kOffRow = kOffStage + NQ * kStage;  // LSE/D row ring: NR x (128 LSE + 128 D) floats
constexpr uint32_t kDSBlock = 2 * kHalf;               // 32 KB
// With stored dS (kStore) the row ring gives up two of its four slots to the
// dS image: this CTA's 128 keys x 128 queries of a tile, [query half][key]
// [64 queries, 128-byte swizzled], the image the dQ kernel loads verbatim.
template <bool kStore>
struct Layout {
  static constexpr int NR = kStore ? 2 : 4;
  static constexpr uint32_t kOffDS = kOffRow + NR * 1024;
  static constexpr uint32_t kOffBar = kOffDS + (kStore ? kDSBlock : 0u);
  static constexpr uint32_t kSmem = kOffBar + 256;
  static_assert(kOffDS % 1024 == 0, "the swizzled dS image starts 1024-byte aligned");
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
};
enum {
  B_KV = 0,                  // K, V landed (even CTA: + the odd CTA's forward)
  B_QFULL = 1,               // NQ: query-half part (Qn, dOn) landed (even CTA: + 1 forward)
  B_QEMPTY = B_QFULL + NQ,   // NQ: query-half part consumed by S^T, dP^T (1 compute thread, this CTA)
  B_HFULL = B_QEMPTY + NQ,   // NQ: head-half part (Qh, dOh) landed (even CTA: + 1 forward)
  B_HEMPTY = B_HFULL + NQ,   // NQ: head-half part consumed by dV, dK (1 compute thread, this CTA)
  B_S = B_HEMPTY + NQ,       // S^T ready (commit, both)
  B_DP = B_S + 1,            // dP^T ready (commit, both)
  B_P = B_DP + 1,            // even CTA: P^T, dS^T written in both CTAs (16 warps)
  B_SFREE = B_P + 1,         // even CTA: S^T copied to registers in both CTAs (16 warps)
  B_DONE = B_SFREE + 1,      // every UMMA done (commit, both)
  B_EPI = B_DONE + 1,        // dK, dV staged (8 warps)
  B_DRAIN = B_EPI + 1,
  B_RFULL = B_DRAIN + 1,     // NR: -LSE/D rows landed (TMA, this CTA)
  // then B_REMPTY (NR): rows read by this CTA's compute warps (8 warps);
  // with stored dS, B_DSFULL: dS of a tile staged (8 warps), and B_DSFREE:
  // the staged dS has been read by its bulk store (store thread)
};
}  // namespace dkdv

template <bool kStore>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ PairParams p) {
  using namespace dkdv;
  constexpr int NR = Layout<kStore>::NR;
  constexpr uint32_t kOffDS = Layout<kStore>::kOffDS, kOffBar = Layout<kStore>::kOffBar;
  constexpr int B_REMPTY = B_RFULL + NR, B_DSFULL = B_REMPTY + NR, B_DSFREE = B_DSFULL + 1;
  constexpr int B_COUNT = B_DSFREE + 1;
  static_assert(8 * B_COUNT + 16 + 12 <= 256, "barriers, TMEM slot and key location fit the barrier area");
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // same condition in both CTAs: both leave before any cluster barrier
    if (threadIdx.x == 0) pair_status(p);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);
  // Where this CTA's keys live, found once at set-up and read back by the
  // producer and the epilogue (computed in both, it would stay live in
  // every warp role).
  int* kv_loc = reinterpret_cast<int*>(smem + kOffBar + 8 * B_COUNT + 16);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  float* rows = reinterpret_cast<float*>(smem + kOffRow);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();

  // Pair work item: (key pair tile, rank, batch, kv head).
  const int pair = blockIdx.x >> 1;
  const int units = p.nranks * p.bs * p.Hk;
  const int np = p.order[pair / units];
  int rest = pair % units;
  const int hk = rest % p.Hk;
  rest /= p.Hk;
  const int b = rest % p.bs;
  const int rl = rest / p.bs;
  const int2 qr = p.range[np];
  const int nm = qr.y - qr.x + 1;
  const int n_it = p.group * nm;
  const int kv0 = np * 256 + 128 * (int)crank;  // this CTA's first key

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_KV || (i >= B_HFULL && i < B_HFULL + NQ) || (i >= B_QFULL && i < B_QFULL + NQ))
        cnt = crank == 0 ? 2 : 1;
      if (i == B_EPI || i == B_DSFULL || (i >= B_REMPTY && i < B_REMPTY + NR)) cnt = 8;
      if (i == B_P || i == B_SFREE) cnt = 16;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hk, hk, kv0);
    kv_loc[0] = l.map;
    kv_loc[1] = l.head;
    kv_loc[2] = l.row;
  }
  if (warp == 9) {
    tmem_alloc2(smem_u32(tmem_slot), 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = p.timeout;

  if (warp >= 8) {
    regs_dec<kRegsOther>();
    if (warp == 8) {
      // --------------------------------------------------------- TMA producer
      bool ok = true;
      // Loads issued so far per ring (rows, query parts, head parts): the
      // last phase armed on slot i of a ring of R slots after c issues is
      // (c - 1 - i) / R, if c > i.
      int n_r = 0, n_q = 0, n_h = 0;
      if (lane == 0) {
        const TileLoc l = {kv_loc[0], kv_loc[1], kv_loc[2]};
        mbar_expect_tx(bar(B_KV), 2 * kTile);
        tma_load_4d(sb + kOffK, &p.ta[l.map], bar(B_KV), 0, l.head, b, l.row);
        tma_load_4d(sb + kOffK + kHalf, &p.ta[l.map], bar(B_KV), 64, l.head, b, l.row);
        tma_load_4d(sb + kOffV, &p.tb[l.map], bar(B_KV), 0, l.head, b, l.row);
        tma_load_4d(sb + kOffV + kHalf, &p.tb[l.map], bar(B_KV), 64, l.head, b, l.row);
      }
      // The head part of tile it-1 is loaded after the query part of tile
      // it: the compute warps free a head part only when they see the dP of
      // the next tile complete (no commit of its own), so it is not needed
      // before then.
      for (int it = 0; it <= n_it; ++it) {
        if (it < n_it) {
          const int st = it % NQ, u = it / NQ;
          const int hq = hk * p.group + it / nm;
          const int q0 = (qr.x + it % nm) * 128;
          const uint32_t sq = sb + kOffStage + st * kStage;
          // query-half part: Q and dO rows [q0 + 64c, +64) (B of S^T, dP^T: N = queries)
          ok = warp_wait(bar(B_QEMPTY + st), (u & 1) ^ 1, lim);
          if (!ok) break;
          if (lane == 0 && !p.skip_q_loads) {
            const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hq, hq, q0);
            const int qh = l.row + 64 * (int)crank;  // the tile's rows are in one shard
            mbar_expect_tx(bar(B_QFULL + st), 2 * kHalf);
            tma_load_4d(sq, &p.tc[l.map], bar(B_QFULL + st), 0, l.head, b, qh);
            tma_load_4d(sq + kHalf / 2, &p.tc[l.map], bar(B_QFULL + st), 64, l.head, b, qh);
            tma_load_4d(sq + kHalf, &p.td[l.map], bar(B_QFULL + st), 0, l.head, b, qh);
            tma_load_4d(sq + kHalf + kHalf / 2, &p.td[l.map], bar(B_QFULL + st), 64, l.head, b, qh);
          }
          n_q = it + 1;
          // -LSE (log2 units) and D of the tile's 128 query rows, one TMA box
          // from the two row planes, needed only once S^T of the tile is
          // done. Rows past sl read as zero; every key masks them, so P = 0
          // there and dS = 0.
          const int rsl = it % NR;
          ok = warp_wait(bar(B_REMPTY + rsl), ((it / NR) & 1) ^ 1, lim);
          if (!ok) break;
          if (lane == 0) {
            mbar_expect_tx(bar(B_RFULL + rsl), 1024);
            tma_load_3d(sb + kOffRow + rsl * 1024, &p.tr[rl], bar(B_RFULL + rsl), q0, b * p.Hq + hq, 0);
          }
          n_r = it + 1;
        }
        if (it >= 1) {
          // head-half part of tile it-1: Q and dO columns [64c, 64c+64) of all 128 rows (B of dK, dV)
          const int ih = it - 1, st = ih % NQ, u = ih / NQ;
          const int hq = hk * p.group + ih / nm;
          const int q0 = (qr.x + ih % nm) * 128;
          const uint32_t sq = sb + kOffStage + st * kStage;
          ok = warp_wait(bar(B_HEMPTY + st), (u & 1) ^ 1, lim);
          if (!ok) break;
          if (lane == 0 && !p.skip_q_loads) {
            const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hq, hq, q0);
            mbar_expect_tx(bar(B_HFULL + st), 2 * kHalf);
            tma_load_4d(sq + 2 * kHalf, &p.te[l.map], bar(B_HFULL + st), 64 * (int)crank, l.head, b, l.row);
            tma_load_4d(sq + 3 * kHalf, &p.tf[l.map], bar(B_HFULL + st), 64 * (int)crank, l.head, b, l.row);
          }
          n_h = ih + 1;
        }
      }
      if (lane == 0) {
        if (!ok) pair_status(p);
        mbar_wait(bar(B_KV), 0, lim);
        for (int i = 0; i < NQ; ++i) {
          if (n_q > i) mbar_wait(bar(B_QFULL + i), ((n_q - 1 - i) / NQ) & 1, lim);
          if (n_h > i) mbar_wait(bar(B_HFULL + i), ((n_h - 1 - i) / NQ) & 1, lim);
        }
        for (int i = 0; i < NR; ++i)
          if (n_r > i) mbar_wait(bar(B_RFULL + i), ((n_r - 1 - i) / NR) & 1, lim);
      }
      __syncwarp();
    } else if (warp == 9 && crank == 0) {
      // --------------------------------------------------------- UMMA issuer (even CTA)
      if (lane == 0) {
        constexpr uint32_t id_kk = idesc_bf16_f32(256, 128, 0, 0);
        constexpr uint32_t id_tm = idesc_bf16_f32(256, 128, 0, 1);
        const uint32_t sK = sb + kOffK, sV = sb + kOffV;
        auto a_kmaj = [](uint32_t base, int kk) {  // 128 rows, K = 128
          return sdesc_sw128(base + (kk >> 2) * kHalf + (kk & 3) * 32, 0, 1024);
        };
        auto b_kmaj64 = [](uint32_t base, int kk) {  // 64 rows, K = 128
          return sdesc_sw128(base + (kk >> 2) * (kHalf / 2) + (kk & 3) * 32, 0, 1024);
        };
        auto b_mn = [](uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, kHalf, 1024); };
        auto issue_s = [&](int st) {
          const uint32_t sq = sb + kOffStage + st * kStage;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) umma2_ss(tmem + 0, a_kmaj(sK, kk), b_kmaj64(sq, kk), id_kk, kk > 0);
        };
        auto issue_dp = [&](int st) {
          const uint32_t sq = sb + kOffStage + st * kStage;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma2_ss(tmem + 128, a_kmaj(sV, kk), b_kmaj64(sq + kHalf, kk), id_kk, kk > 0);
        };
        bool ok = mbar_wait(bar(B_KV), 0, lim) && mbar_wait(bar(B_QFULL), 0, lim);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          umma2_commit_both(bar(B_S));
          issue_dp(0);
          umma2_commit_both(bar(B_DP));
        }
        if (ok && n_it > 1) {
          ok = mbar_wait(bar(B_SFREE), 0, lim) && mbar_wait(bar(B_QFULL + 1 % NQ), (1 / NQ) & 1, lim);
          if (ok) {
            tc_fence_after();
            issue_s(1 % NQ);
            umma2_commit_both(bar(B_S));
          }
        }
        // Per query tile i, in issue order:
        //   dV += P_i^T dO_i and dK += dS_i^T Q_i, interleaved, once P_i is written;
        //   dP_{i+1}^T, over P_i^T and dS_i^T (after dV and dK have read them);
        //   S_{i+2}^T, over S_{i+1}^T, once the compute warps have copied that out.
        // So S_{i+2} runs while the compute warps turn dP_{i+1} into dS_{i+1},
        // and the exponentials of tile i+1 overlap dV_i, dK_i and dP_{i+1}.
        for (int it = 0; it < n_it && ok; ++it) {
          const int st = it % NQ;
          const uint32_t sq = sb + kOffStage + st * kStage;
          if (!mbar_wait(bar(B_P), it & 1, lim) || !mbar_wait(bar(B_HFULL + st), (it / NQ) & 1, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dV += P^T dO and dK += dS^T Q, interleaved
            // query half kk/4 of P^T at 128 + 64 (kk/4), of dS^T 32 columns further
            const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
            const uint32_t a = tmem + 128 + (kk >> 2) * 64 + (kk & 3) * 8;
            umma2_ts(tmem + 256, a, b_mn(sq + 3 * kHalf, kk), id_tm, acc);
            umma2_ts(tmem + 384, a + 32, b_mn(sq + 2 * kHalf, kk), id_tm, acc);
          }
          if (it + 1 < n_it) {
            issue_dp((it + 1) % NQ);  // its query part landed before S_{i+1} was issued
            umma2_commit_both(bar(B_DP));
          }
          if (it + 2 < n_it) {
            const int st2 = (it + 2) % NQ;
            if (!mbar_wait(bar(B_SFREE), (it + 1) & 1, lim) ||
                !mbar_wait(bar(B_QFULL + st2), ((it + 2) / NQ) & 1, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(st2);
            umma2_commit_both(bar(B_S));
          }
        }
        if (ok)
          umma2_commit_both(bar(B_DONE));
        else
          pair_status(p);
        umma2_commit_both(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, lim);
      }
      __syncwarp();
    } else if (warp == 10 && crank == 1) {
      // --------------------------------------------------------- forwarder (odd CTA)
      // The even CTA's UMMAs read this CTA's shared memory: tell it when the
      // loads have landed.
      if (lane == 0) {
        bool ok = mbar_wait(bar(B_KV), 0, lim);
        if (ok) mbar_arrive_cluster(mapa(bar(B_KV), 0));
        for (int it = 0; it <= n_it && ok; ++it) {  // in the producer's order
          if (it < n_it) {
            const int st = it % NQ, u = it / NQ;
            ok = mbar_wait(bar(B_QFULL + st), u & 1, lim);
            if (ok) mbar_arrive_cluster(mapa(bar(B_QFULL + st), 0));
          }
          if (ok && it >= 1) {
            const int st = (it - 1) % NQ, u = (it - 1) / NQ;
            ok = mbar_wait(bar(B_HFULL + st), u & 1, lim);
            if (ok) mbar_arrive_cluster(mapa(bar(B_HFULL + st), 0));
          }
        }
        if (!ok) pair_status(p);
      }
      __syncwarp();
    } else if (kStore && warp == 11) {
      // --------------------------------------------------------- dS store (both CTAs)
      // Block (key pair np, query tile m) of a (rank, batch, head) is 64 KB:
      // the even CTA's 32 KB image, then the odd CTA's.
      if (lane == 0) {
        const uint64_t pol = l2_evict_first();
        const long long first = p.ds_base[np];
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
          if (!mbar_wait(bar(B_DSFULL), it & 1, lim)) {
            ok = false;
            break;
          }
          const int hq = hk * p.group + it / nm;
          const long long blk = ((long long)(rl * p.bs + b) * p.Hq + hq) * p.ds_nblk + first + it % nm;
          bulk_store(p.ds + (size_t)(2 * blk + crank) * kDSBlock, sb + kOffDS, kDSBlock, pol);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(bar(B_DSFREE));
        }
        if (!ok) pair_status(p);
      }
      __syncwarp();
    }
  } else {
    regs_inc<kRegsCompute>();
    // ----------------------------------------------------------- compute warps
    const int quarter = warp & 3;
    const int h = warp >> 2;                 // query half: columns [64h, 64h+64)
    const int jr = quarter * 32 + lane;      // key row within this CTA = TMEM lane
    const int j = kv0 + jr;                  // global key position
    int qlo = 1, qhi = 0;                    // queries that see key j: [qlo, qhi]
    if (j < p.sl) {
      const int d = doc_of(p.doc_offsets, p.ndoc, j);
      qlo = p.causal ? j : p.doc_offsets[d];
      qhi = p.doc_offsets[d + 1] - 1;
    }
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int m = qr.x + it % nm;
      const int rsl = it % NR;
      ok = warp_wait(bar(B_S), it & 1, lim);
      ok = ok && warp_wait(bar(B_RFULL + rsl), (it / NR) & 1, lim);
      if (!ok) break;
      tc_fence_after();
      uint32_t pf[64];
      tmem_ld32(tmem + lane_base + 0 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pf[0]));
      tmem_ld32(tmem + lane_base + 32 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pf[32]));
      tmem_ld_wait(pf);
      tc_fence_before();
      warp_arrive_leader(bar(B_SFREE), crank);  // S^T may be overwritten by S of tile it+2
      const float* rs = rows + rsl * 256;
      const int i0 = m * 128 + 64 * h;
      const bool full = qlo <= i0 && i0 + 63 <= qhi;
      // P^T = 2^(S^T * scale*log2(e) - LSE), two query columns per packed op
      const uint64_t sc2 = f2(sl2, sl2);
      const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(rs + 64 * h);
      uint64_t pp[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pp[c] = f2_ex2(f2_fma(f2_bits(pf[2 * c], pf[2 * c + 1]), sc2, nl2[c]));
      if (!full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float p0, p1;
          f2_split(pp[c], p0, p1);
          const int i = i0 + 2 * c;
          if (i < qlo || i > qhi) p0 = 0.f;
          if (i + 1 < qlo || i + 1 > qhi) p1 = 0.f;
          pp[c] = f2(p0, p1);
        }
      }
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = f2_pack_bf16(pp[c]);
      ok = warp_wait(bar(B_DP), it & 1, lim);
      if (!ok) break;
      tc_fence_after();
      if (warp == 0 && lane == 0) {
        // dP^T of tile it has completed, and with it S^T: the query part of
        // its stage is free for the producer. dV and dK of tile it-1 were
        // issued before this dP, so they have completed too: the head part
        // of that tile's stage is free.
        mbar_arrive(bar(B_QEMPTY + it % NQ));
        if (it > 0) mbar_arrive(bar(B_HEMPTY + (it - 1) % NQ));
      }
      __syncwarp();
      uint32_t dp[64];
      tmem_ld32(tmem + lane_base + 128 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tmem + lane_base + 160 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_ld_wait(dp);
      // P^T and dS^T (bf16) over the dP^T columns this thread has just read
      // (no other thread reads them); the store of P^T runs while dS^T is
      // formed.
      tmem_st32(tmem + lane_base + 128 + 64 * h, pk);
      // dS^T = P^T * (dP^T - D)
      const uint64_t* d2 = reinterpret_cast<const uint64_t*>(rs + 128 + 64 * h);
      uint32_t dk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) dk[c] = f2_pack_bf16(f2_mul(pp[c], f2_sub(f2_bits(dp[2 * c], dp[2 * c + 1]), d2[c])));
      tmem_st32(tmem + lane_base + 160 + 64 * h, dk);
      tmem_st_wait(pk);
      tc_fence_before();
      warp_arrive_leader(bar(B_P), crank);
      // Done with this tile's LSE/D rows. The producer refills the slot by
      // TMA (the async proxy) once every warp has arrived: the proxy fence
      // orders this thread's generic reads of the slot before that write.
      fence_proxy_async_smem();
      warp_arrive_local(bar(B_REMPTY + rsl));
      if (kStore) {
        // dS^T row jr = column jr of dS, staged for the store thread once it
        // has read the previous tile's image out.
        ok = warp_wait(bar(B_DSFREE), (it & 1) ^ 1, lim);
        if (!ok) break;
        stage_row64(sb + kOffDS + h * kHalf, jr, dk);
        fence_proxy_async_smem();
        warp_arrive_local(bar(B_DSFULL));
      }
    }
    if (ok) ok = warp_wait(bar(B_DONE), 0, lim);
    if (ok) {
      tc_fence_after();
      // dV (columns 256+) and dK (384+, times s) of key row jr, head-dimension
      // half h, staged in this CTA's V and K tiles (free now) and TMA-stored.
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t col = (which == 0 ? 256 : 384) + 64 * h;
        uint32_t o[64], w[32];
        tmem_ld32(tmem + lane_base + col, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tmem_ld32(tmem + lane_base + col + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tmem_ld_wait(o);
#pragma unroll
        for (int c = 0; c < 32; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * mul, __uint_as_float(o[2 * c + 1]) * mul);
        stage_row64(sb + (which == 0 ? kOffV : kOffK) + h * kHalf, jr, w);
      }
      fence_proxy_async_smem();
      warp_arrive_local(bar(B_EPI));
      if (threadIdx.x == 0) {
        if (mbar_wait(bar(B_EPI), 0, lim)) {
          const TileLoc l = {kv_loc[0], kv_loc[1], kv_loc[2]};
          tma_store_4d(&p.th[l.map], sb + kOffV, 0, l.head, b, l.row);
          tma_store_4d(&p.th[l.map], sb + kOffV + kHalf, 64, l.head, b, l.row);
          tma_store_4d(&p.tg[l.map], sb + kOffK, 0, l.head, b, l.row);
          tma_store_4d(&p.tg[l.map], sb + kOffK + kHalf, 64, l.head, b, l.row);
          bulk_commit();
          bulk_wait_read_all();  // the stores have read shared memory; their global writes complete before the grid does
        } else {
          pair_status(p);
        }
      }
    } else if (lane == 0) {
      pair_status(p);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or multicast commit can target an exited CTA
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc2(tmem, 512);
  }
}

// ===========================================================================
// dQ: pair = 256 queries
// ===========================================================================
namespace dqk {
constexpr int NK = 3;
constexpr uint32_t kOffQ = 0, kOffDO = kTile;
// Per stage: Kn, Vn (this CTA's 64 key rows x 128, K-major), then Kh (all 128
// key rows x this CTA's 64 head columns, MN-major).
constexpr uint32_t kOffStage = 2 * kTile;
constexpr uint32_t kStage = 3 * kHalf;
constexpr uint32_t kOffBar = kOffStage + NK * kStage;
constexpr uint32_t kSmem = kOffBar + 256;
enum {
  B_QO = 0,                  // Q, dO landed (even CTA: + forward)
  B_KFULL = 1,               // NK: key stage landed (even CTA: + forward)
  B_KEMPTY = B_KFULL + NK,   // NK: key stage consumed: dQ of its tile done (commit, both)
  B_DP = B_KEMPTY + NK,      // S and dP of a tile ready (commit after dP, both)
  B_SFREE = B_DP + 1,        // even CTA: S copied out of tensor memory in both CTAs (16 warps)
  B_DS = B_SFREE + 1,        // even CTA: dS written in both CTAs (16 warps)
  B_DONE = B_DS + 1,         // every UMMA done (commit, both)
  B_EPI = B_DONE + 1,        // dQ staged (8 warps)
  B_DRAIN = B_EPI + 1,
  B_COUNT
};
}  // namespace dqk

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ PairParams p) {
  using namespace dqk;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {
    if (threadIdx.x == 0) pair_status(p);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();

  // Pair work item: (query pair tile, rank, batch, query head).
  const int pair = blockIdx.x >> 1;
  const int units = p.nranks * p.bs * p.Hq;
  const int mp = p.order[pair / units];
  int rest = pair % units;
  const int hq = rest % p.Hq;
  rest /= p.Hq;
  const int b = rest % p.bs;
  const int rl = rest / p.bs;
  const int hk = hq / p.group;
  const int2 kr = p.range[mp];
  const int n_kv = kr.y - kr.x + 1;
  const int q0 = mp * 256 + 128 * (int)crank;  // this CTA's first query

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_QO || (i >= B_KFULL && i < B_KFULL + NK)) cnt = crank == 0 ? 2 : 1;
      if (i == B_EPI) cnt = 8;
      if (i == B_DS || i == B_SFREE) cnt = 16;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc2(smem_u32(tmem_slot), 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = p.timeout;
  // Tensor memory: S in [0,128); dP of tile j in buffer j&1, [128,256) or
  // [256,384), with dS (bf16) written over the buffer's columns [0,32) and
  // [64,96); the dQ accumulator in [384,512).

  if (warp >= 8) {
    regs_dec<kRegsOther>();
    if (warp == 8) {
      // --------------------------------------------------------- TMA producer
      if (lane == 0) {
        bool ok = true;
        int last[NK];
        for (int i = 0; i < NK; ++i) last[i] = -1;
        const TileLoc lq = locate_tile(p.fused, p.n, p.nranks, rl, p.Hq, hq, q0);
        mbar_expect_tx(bar(B_QO), 2 * kTile);
        tma_load_4d(sb + kOffQ, &p.ta[lq.map], bar(B_QO), 0, lq.head, b, lq.row);
        tma_load_4d(sb + kOffQ + kHalf, &p.ta[lq.map], bar(B_QO), 64, lq.head, b, lq.row);
        tma_load_4d(sb + kOffDO, &p.tb[lq.map], bar(B_QO), 0, lq.head, b, lq.row);
        tma_load_4d(sb + kOffDO + kHalf, &p.tb[lq.map], bar(B_QO), 64, lq.head, b, lq.row);
        for (int jj = 0; jj < n_kv; ++jj) {
          const int st = jj % NK, u = jj / NK;
          const int k0 = (kr.x + jj) * 128;
          if (!mbar_wait(bar(B_KEMPTY + st), (u & 1) ^ 1, lim)) { ok = false; break; }
          const uint32_t sk = sb + kOffStage + st * kStage;
          mbar_expect_tx(bar(B_KFULL + st), 3 * kHalf);
          // key half of K and V (B of S, dP: N = keys); the tile's keys are in one shard
          const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hk, hk, k0);
          const int rn = l.row + 64 * (int)crank;
          tma_load_4d(sk, &p.tc[l.map], bar(B_KFULL + st), 0, l.head, b, rn);
          tma_load_4d(sk + kHalf / 2, &p.tc[l.map], bar(B_KFULL + st), 64, l.head, b, rn);
          tma_load_4d(sk + kHalf, &p.td[l.map], bar(B_KFULL + st), 0, l.head, b, rn);
          tma_load_4d(sk + kHalf + kHalf / 2, &p.td[l.map], bar(B_KFULL + st), 64, l.head, b, rn);
          // head-dimension half of K (B of dQ: N = head dimension)
          tma_load_4d(sk + 2 * kHalf, &p.te[l.map], bar(B_KFULL + st), 64 * (int)crank, l.head, b, l.row);
          last[st] = u;
        }
        if (!ok) pair_status(p);
        mbar_wait(bar(B_QO), 0, lim);
        for (int i = 0; i < NK; ++i)
          if (last[i] >= 0) mbar_wait(bar(B_KFULL + i), last[i] & 1, lim);
      }
      __syncwarp();
    } else if (warp == 9 && crank == 0) {
      // --------------------------------------------------------- UMMA issuer (even CTA)
      if (lane == 0) {
        constexpr uint32_t id_kk = idesc_bf16_f32(256, 128, 0, 0);
        constexpr uint32_t id_tm = idesc_bf16_f32(256, 128, 0, 1);
        // Descriptors are formed once per operand and stepped by constants,
        // so that each UMMA costs the issuing thread one add.
        auto kmaj = [](uint32_t base) { return sdesc_sw128(base, 0, 1024); };
        auto a_kmaj = [](uint64_t d, int kk) { return sdesc_add(d, (kk >> 2) * kHalf + (kk & 3) * 32); };
        auto b_kmaj64 = [](uint64_t d, int kk) { return sdesc_add(d, (kk >> 2) * (kHalf / 2) + (kk & 3) * 32); };
        auto b_mn = [](uint64_t d, int kk) { return sdesc_add(d, kk * 2048); };
        auto issue_s = [&](int jj) {
          const uint64_t dq = kmaj(sb + kOffQ), dk = kmaj(sb + kOffStage + (jj % NK) * kStage);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) umma2_ss(tmem + 0, a_kmaj(dq, kk), b_kmaj64(dk, kk), id_kk, kk > 0);
        };
        // dP of tile jj into buffer jj&1; its commit also covers S of the tile.
        auto issue_dp = [&](int jj) {
          const uint64_t ddo = kmaj(sb + kOffDO), dv = kmaj(sb + kOffStage + (jj % NK) * kStage + kHalf);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma2_ss(tmem + 128 + 128 * (jj & 1), a_kmaj(ddo, kk), b_kmaj64(dv, kk), id_kk, kk > 0);
          umma2_commit_both(bar(B_DP));
        };
        bool ok = mbar_wait(bar(B_QO), 0, lim) && mbar_wait(bar(B_KFULL), 0, lim);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
        // Per key tile jj, in issue order: S and dP of tile jj+1 (once the
        // compute warps have copied S of tile jj out), then dQ += dS K of
        // tile jj once its dS is written. The tensor pipe thus runs the next
        // tile's S and dP while the compute warps form this tile's dS.
        for (int jj = 0; jj < n_kv && ok; ++jj) {
          const int st = jj % NK;
          if (jj + 1 < n_kv) {
            const int st1 = (jj + 1) % NK, u1 = (jj + 1) / NK;
            if (!mbar_wait(bar(B_KFULL + st1), u1 & 1, lim) || !mbar_wait(bar(B_SFREE), jj & 1, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(jj + 1);
            issue_dp(jj + 1);  // buffer (jj+1)&1: its dS was read by dQ of tile jj-1, issued before
          }
          if (!mbar_wait(bar(B_DS), jj & 1, lim)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dkh = sdesc_sw128(sb + kOffStage + st * kStage + 2 * kHalf, kHalf, 1024);
          const uint32_t ds = tmem + 128 + 128 * (jj & 1);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ += dS K; key half kk/4 of dS at +64 (kk/4)
            umma2_ts(tmem + 384, ds + (kk >> 2) * 64 + (kk & 3) * 8, b_mn(dkh, kk), id_tm,
                     (jj > 0 || kk > 0) ? 1u : 0u);
          umma2_commit_both(bar(B_KEMPTY + st));  // the key stage is free once dQ has read it
        }
        if (ok)
          umma2_commit_both(bar(B_DONE));
        else
          pair_status(p);
        umma2_commit_both(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, lim);
      }
      __syncwarp();
    } else if (warp == 10 && crank == 1) {
      // --------------------------------------------------------- forwarder (odd CTA)
      if (lane == 0) {
        bool ok = mbar_wait(bar(B_QO), 0, lim);
        if (ok) mbar_arrive_cluster(mapa(bar(B_QO), 0));
        for (int jj = 0; jj < n_kv && ok; ++jj) {
          const int st = jj % NK, u = jj / NK;
          ok = mbar_wait(bar(B_KFULL + st), u & 1, lim);
          if (ok) mbar_arrive_cluster(mapa(bar(B_KFULL + st), 0));
        }
        if (!ok) pair_status(p);
      }
      __syncwarp();
    }
  } else {
    regs_inc<kRegsCompute>();
    // ----------------------------------------------------------- compute warps
    const int quarter = warp & 3;
    const int h = warp >> 2;                 // key half: columns [64h, 64h+64)
    const int iq = quarter * 32 + lane;      // query row within this CTA = TMEM lane
    const int i = q0 + iq;                   // global query position
    int klo = 1, khi = 0;                    // keys visible from query i: [klo, khi]
    float nl2 = -INFINITY, Di = 0.f;  // -LSE (log2 units) and D of row i
    if (i < p.sl) {
      const int d = doc_of(p.doc_offsets, p.ndoc, i);
      klo = p.doc_offsets[d];
      khi = p.causal ? i : p.doc_offsets[d + 1] - 1;
      const size_t plane = (size_t)p.bs * p.Hq * p.pitch;
      const size_t base = ((size_t)b * p.Hq + hq) * p.pitch + i;
      nl2 = p.rows[rl][base];
      Di = p.rows[rl][plane + base];
    }
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint64_t sc2 = f2(p.scale_log2, p.scale_log2), nlp = f2(nl2, nl2), D2 = f2(Di, Di);
    // The even CTA's barriers in the cluster's shared window (its own, for the
    // even CTA), computed once: a per-arrive branch on the CTA rank made the
    // compiler spill while S is held in registers.
    const uint32_t sfree_c = mapa(bar(B_SFREE), 0), ds_c = mapa(bar(B_DS), 0);
    bool ok = true;
    for (int jj = 0; jj < n_kv; ++jj) {
      const int k0 = (kr.x + jj) * 128 + 64 * h;
      ok = warp_wait(bar(B_DP), jj & 1, lim);
      if (!ok) break;
      tc_fence_after();
      uint32_t pf[64];
      tmem_ld32(tmem + lane_base + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pf[0]));
      tmem_ld32(tmem + lane_base + 32 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&pf[32]));
      tmem_ld_wait(pf);
      tc_fence_before();
      warp_arrive_cluster(sfree_c);  // S may be overwritten by S of tile jj+1
      const bool full = klo <= k0 && k0 + 63 <= khi;
      uint64_t pp[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pp[c] = f2_ex2(f2_fma(f2_bits(pf[2 * c], pf[2 * c + 1]), sc2, nlp));
      if (!full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float p0, p1;
          f2_split(pp[c], p0, p1);
          const int key = k0 + 2 * c;
          if (key < klo || key > khi) p0 = 0.f;
          if (key + 1 < klo || key + 1 > khi) p1 = 0.f;
          pp[c] = f2(p0, p1);
        }
      }
      const uint32_t dpb = tmem + lane_base + 128 + 128 * (jj & 1) + 64 * h;
      uint32_t dp[64];
      tmem_ld32(dpb, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(dpb + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_ld_wait(dp);
      uint32_t dk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) dk[c] = f2_pack_bf16(f2_mul(pp[c], f2_sub(f2_bits(dp[2 * c], dp[2 * c + 1]), D2)));
      tmem_st32(dpb, dk);  // dS (bf16) over the dP columns this thread read
      tmem_st_wait();
      tc_fence_before();
      warp_arrive_cluster(ds_c);
    }
    if (ok) ok = warp_wait(bar(B_DONE), 0, lim);
    if (ok) {
      tc_fence_after();
      // dQ (times s) of query row iq, head-dimension half h, staged in the Q
      // tile (free now) and TMA-stored.
      uint32_t o[64], w[32];
      tmem_ld32(tmem + lane_base + 384 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
      tmem_ld32(tmem + lane_base + 416 + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
      tmem_ld_wait(o);
#pragma unroll
      for (int c = 0; c < 32; ++c)
        w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * p.scale, __uint_as_float(o[2 * c + 1]) * p.scale);
      stage_row64(sb + kOffQ + h * kHalf, iq, w);
      fence_proxy_async_smem();
      warp_arrive_local(bar(B_EPI));
      if (threadIdx.x == 0) {
        if (mbar_wait(bar(B_EPI), 0, lim)) {
          const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hq, hq, q0);
          tma_store_4d(&p.tf[l.map], sb + kOffQ, 0, l.head, b, l.row);
          tma_store_4d(&p.tf[l.map], sb + kOffQ + kHalf, 64, l.head, b, l.row);
          bulk_commit();
          bulk_wait_read_all();  // the stores have read shared memory; their global writes complete before the grid does
        } else {
          pair_status(p);
        }
      }
    } else if (lane == 0) {
      pair_status(p);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc2(tmem, 512);
  }
}

// ===========================================================================
// dQ from stored dS: pair = 256 queries
// ===========================================================================
// When the dK/dV kernel has written dS to the workspace, dQ = s dS K is one
// GEMM per (query tile, key tile): the CTA pair streams the dS images of its
// two query tiles (the A operand, MN-major: queries contiguous) and the key
// tiles' head-dimension halves (B, MN-major) through a ring of stages, with
// M = 256 UMMAs into one tensor-memory accumulator. No exponentials, no
// masks: a block the dK/dV kernel did not visit holds no visible pair, and
// reads 32 KB of zeros instead.
namespace dqs {
constexpr int kThreads = 192;
constexpr int NS = 4;
constexpr uint32_t kDS = 2 * kHalf;            // dS image: [query half][128 keys][64 queries], 32 KB
constexpr uint32_t kStage = kDS + kHalf;       // + K: [128 keys][this CTA's 64 head columns], 16 KB
constexpr uint32_t kOffBar = NS * kStage;
constexpr uint32_t kSmem = kOffBar + 256;
static_assert(kStage % 1024 == 0 && kSmem <= 227 * 1024, "stages 1024-byte aligned, within shared memory");
enum {
  B_FULL = 0,                // NS: dS image and K landed (even CTA: + forward)
  B_EMPTY = B_FULL + NS,     // NS: stage read by its UMMAs (commit, both)
  B_DONE = B_EMPTY + NS,     // every UMMA done (commit, both)
  B_EPI = B_DONE + 1,        // dQ staged (4 warps)
  B_DRAIN = B_EPI + 1,
  B_COUNT
};
}  // namespace dqs

struct DqsParams {
  CUtensorMap tk[kRanksPerLaunch];   // K, boxes of 64 head columns x 128 rows
  CUtensorMap tq[kRanksPerLaunch];   // dQ (store), boxes of 64 x 128
  const int2* range;                 // per query pair tile: first and last key tile
  const int* order;                  // query pair tiles, most work first
  const int2* kv_range;              // per key pair tile: the query tiles holding stored blocks
  const int* ds_base;                // per key pair tile: its first block in a (rank, batch, head)
  const char* ds;                    // blocks of the launch's first rank
  const char* zero;                  // 32 KB of zeros
  long long ds_nblk;                 // blocks per (rank, batch, head)
  unsigned* status;
  long long timeout;
  int bs, Hq, Hk, group, nranks, fused, n;
  float scale;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(dqs::kThreads, 1)
    attn_bwd_dq_stored_kernel(const __grid_constant__ DqsParams p) {
  using namespace dqs;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, STATUS_TIMEOUT);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto fail = [&]() { atomicOr(p.status, STATUS_TIMEOUT); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();

  // Pair work item: (query pair tile, rank, batch, query head).
  const int pair = blockIdx.x >> 1;
  const int units = p.nranks * p.bs * p.Hq;
  const int mp = p.order[pair / units];
  int rest = pair % units;
  const int hq = rest % p.Hq;
  rest /= p.Hq;
  const int b = rest % p.bs;
  const int rl = rest / p.bs;
  const int hk = hq / p.group;
  const int2 kr = p.range[mp];
  const int n_kv = kr.y - kr.x + 1;
  const int m = 2 * mp + (int)crank;  // this CTA's query tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i >= B_FULL && i < B_FULL + NS) cnt = crank == 0 ? 2 : 1;
      if (i == B_EPI) cnt = 4;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc2(smem_u32(tmem_slot), 128);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = p.timeout;

  if (warp == 4) {
    // ----------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      const long long unit = (long long)(rl * p.bs + b) * p.Hq + hq;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % NS, u = j / NS;
        if (!mbar_wait(bar(B_EMPTY + st), (u & 1) ^ 1, lim)) {
          ok = false;
          break;
        }
        const int kt = kr.x + j, np = kt >> 1;
        const int2 qr = p.kv_range[np];
        const char* src = p.zero;
        if (m >= qr.x && m <= qr.y)
          src = p.ds + (size_t)(2 * (unit * p.ds_nblk + p.ds_base[np] + (m - qr.x)) + (kt & 1)) * kDS;
        const uint32_t sst = sb + st * kStage;
        mbar_expect_tx(bar(B_FULL + st), kStage);
        bulk_load(sst, src, kDS, bar(B_FULL + st), pol);
        const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hk, hk, kt * 128);
        tma_load_4d(sst + kDS, &p.tk[l.map], bar(B_FULL + st), 64 * (int)crank, l.head, b, l.row);
      }
      if (!ok) fail();
      for (int i = 0; i < NS; ++i)  // no copy in flight at exit
        if (n_kv > i) mbar_wait(bar(B_FULL + i), ((n_kv - 1 - i) / NS) & 1, lim);
    }
    __syncwarp();
  } else if (warp == 5 && crank == 0) {
    // ----------------------------------------------------------- UMMA issuer (even CTA)
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16_f32(256, 128, 1, 1);
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % NS, u = j / NS;
        if (!mbar_wait(bar(B_FULL + st), u & 1, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sst = sb + st * kStage;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // keys [16kk, 16kk+16): 16 rows of 128 bytes in both operands
          umma2_ss(tmem, sdesc_sw128(sst + kk * 2048, kHalf, 1024), sdesc_sw128(sst + kDS + kk * 2048, kHalf, 1024),
                   id, (j > 0 || kk > 0) ? 1u : 0u);
        umma2_commit_both(bar(B_EMPTY + st));
      }
      if (ok)
        umma2_commit_both(bar(B_DONE));
      else
        fail();
      umma2_commit_both(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, lim);
    }
    __syncwarp();
  } else if (warp == 5 && crank == 1) {
    // ----------------------------------------------------------- forwarder (odd CTA)
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int st = j % NS, u = j / NS;
        ok = mbar_wait(bar(B_FULL + st), u & 1, lim);
        if (ok) mbar_arrive_cluster(mapa(bar(B_FULL + st), 0));
      }
      if (!ok) fail();
    }
    __syncwarp();
  } else if (warp < 4) {
    // ----------------------------------------------------------- epilogue
    // dQ (times s) of query row iq, staged in stage 0 (free once every UMMA
    // is done) as two 64-column halves and TMA-stored.
    const int iq = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const bool ok = warp_wait(bar(B_DONE), 0, lim);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o[64], w[32];
        tmem_ld32(tmem + lane_base + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tmem_ld32(tmem + lane_base + 64 * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tmem_ld_wait(o);
#pragma unroll
        for (int c = 0; c < 32; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * p.scale, __uint_as_float(o[2 * c + 1]) * p.scale);
        stage_row64(sb + hh * kHalf, iq, w);
      }
      fence_proxy_async_smem();
      warp_arrive_local(bar(B_EPI));
      if (threadIdx.x == 0) {
        if (mbar_wait(bar(B_EPI), 0, lim)) {
          const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hq, hq, m * 128);
          tma_store_4d(&p.tq[l.map], sb, 0, l.head, b, l.row);
          tma_store_4d(&p.tq[l.map], sb + kHalf, 64, l.head, b, l.row);
          bulk_commit();
          bulk_wait_read_all();
        } else {
          fail();
        }
      }
    } else if (lane == 0) {
      fail();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc2(tmem, 128);
  }
}

// The row planes of the backward, for every (rank, batch, head, row):
// -LSE * log2(e) (plane 0) and D = rowsum(dO * O) (plane 1), each
// [bs][Hq][pitch] fp32. 16 lanes per row. O and dO are head shards, or
// sequence shards when fused (row t of rank r's head hq is then token
// t - s*n of shard s = t / n, head r*Hq + hq).
struct PrepParams {
  const __nv_bfloat16* o[ULYSSES_MAX_P];
  const __nv_bfloat16* dO[ULYSSES_MAX_P];
  const float* lse[ULYSSES_MAX_P];
  float* rows[ULYSSES_MAX_P];
  uint4* zero;                       // 32 KB to clear (the stored-dS zero block), or null
  int P, sl, bs, Hq, pitch;
  int fused, n;
};

// Rows are taken in the memory order of the buffers that hold O and dO, so
// every block streams 64 consecutive 256-byte rows (16 KB) of each: buffer i
// holds rows rho = (t*bs + b)*Hq + hq of head shard i, or, fused, rows
// rho = (tt*bs + b)*hc + h of sequence shard i (token t = i*n + tt, rank
// h / Hq, head h % Hq). Both have sl*bs*Hq rows. Warp w takes rows
// [8w, 8w+8) of the block in four steps of two rows, a half-warp (16 lanes
// x 16 bytes of O and of dO) per row, with all eight loads of a lane issued
// before the first sum. grid.x covers the rows of a buffer, grid.y the
// buffers.
constexpr int kPrepRows = 64;
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const __grid_constant__ PrepParams a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, part = lane & 15;
  const int src = blockIdx.y;
  const long long nrows = (long long)a.sl * a.bs * a.Hq;
  const long long rho0 = (long long)blockIdx.x * kPrepRows + warp * 8;
  if (a.zero && blockIdx.x == 0 && blockIdx.y == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) a.zero[i * 256 + threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  }
  {
    uint4 ov[4], dv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long rho = rho0 + 2 * u + half;
      ov[u] = dv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (rho < nrows) {
        ov[u] = __ldg(reinterpret_cast<const uint4*>(a.o[src] + rho * 128) + part);
        dv[u] = __ldg(reinterpret_cast<const uint4*>(a.dO[src] + rho * 128) + part);
      }
    }
    float acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[u]);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv[u]);
      float x = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(o2[e]);
        const float2 df = __bfloat1622float2(d2[e]);
        x = fmaf(of.x, df.x, fmaf(of.y, df.y, x));
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      acc[u] = x;  // the sum of row 2u + half, in every lane of the half
    }
    // D of row j (0..7) to lane j: row j is step j/2 of half j%2.
    float d = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float v0 = __shfl_sync(0xffffffffu, acc[u], 0), v1 = __shfl_sync(0xffffffffu, acc[u], 16);
      if (lane == 2 * u) d = v0;
      if (lane == 2 * u + 1) d = v1;
    }
    // Lanes 0-7 write D of rows rho0 + lane, lanes 8-15 the -LSE log2(e) of
    // rows rho0 + lane - 8.
    const long long rho = rho0 + (lane & 7);
    if (lane < 16 && rho < nrows) {
      int t, b, r, hq;
      if (a.fused) {
        const int hc = a.P * a.Hq;
        const int h = (int)(rho % hc);
        b = (int)((rho / hc) % a.bs);
        t = src * a.n + (int)(rho / ((long long)hc * a.bs));
        r = h / a.Hq;
        hq = h % a.Hq;
      } else {
        hq = (int)(rho % a.Hq);
        b = (int)((rho / a.Hq) % a.bs);
        t = (int)(rho / ((long long)a.Hq * a.bs));
        r = src;
      }
      const size_t row = ((size_t)b * a.Hq + hq) * a.pitch + t;
      if (lane < 8)
        a.rows[r][(size_t)a.bs * a.Hq * a.pitch + row] = d;
      else
        a.rows[r][row] = -(a.lse[r][((size_t)b * a.Hq + hq) * a.sl + t] * 1.4426950408889634f);
    }
  }
}

}  // namespace

// Pair schedules. dK/dV: per 256-key pair tile, the range of 128-row query
// tiles that can see any of its keys. Forward and dQ: per 256-query pair
// tile, the range of 128-key tiles any of its queries can see. Both ordered
// by work, most first.
void plan_pair_tiles(const Layer& L, std::vector<int2>& kv_pairs, std::vector<int>& kv_order,
                     std::vector<int2>& q_pairs, std::vector<int>& q_order) {
  const int sl = (int)L.sl;
  const int n_pair = (sl + 255) / 256;
  auto doc = [&](int t) {
    return (int)(std::upper_bound(L.doc_offsets.begin(), L.doc_offsets.end(), t) - L.doc_offsets.begin()) - 1;
  };
  auto order_by = [](const std::vector<int2>& r, std::vector<int>& order) {
    order.resize(r.size());
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int c) { return r[a].y - r[a].x > r[c].y - r[c].x; });
  };
  kv_pairs.resize(n_pair);
  q_pairs.resize(n_pair);
  for (int t = 0; t < n_pair; ++t) {
    const int first = t * 256, last = std::min(sl, first + 256) - 1;
    // keys [first, last]: the queries that see them
    const int lo_q = L.causal ? first : L.doc_offsets[doc(first)];
    const int hi_q = L.doc_offsets[doc(last) + 1] - 1;
    kv_pairs[t] = make_int2(lo_q / 128, hi_q / 128);
    // queries [first, last]: the keys they see
    const int lo_k = L.doc_offsets[doc(first)];
    const int hi_k = L.causal ? last : L.doc_offsets[doc(last) + 1] - 1;
    q_pairs[t] = make_int2(lo_k / 128, hi_k / 128);
  }
  order_by(kv_pairs, kv_order);
  order_by(q_pairs, q_order);
}

int64_t plan_ds_blocks(const std::vector<int2>& kv_pairs, std::vector<int>& base) {
  base.resize(kv_pairs.size());
  int64_t n = 0;
  for (size_t t = 0; t < kv_pairs.size(); ++t) {
    base[t] = (int)n;
    n += kv_pairs[t].y - kv_pairs[t].x + 1;
  }
  return n;
}

int64_t bwd_row_pitch(const Layer& L) { return (L.sl + 3) / 4 * 4; }
size_t bwd_sm103_workspace(const Layer& L) { return (size_t)L.P * 2 * L.bs * L.Hq * bwd_row_pitch(L) * sizeof(float); }
// The stored-dS area starts after the row planes of the capacity, so its
// place does not move with the sequence: first a 32 KB zero block, then per
// (rank, batch, head) nblk blocks of 64 KB.
size_t bwd_ds_offset(const Layer& L) {
  const size_t rows = (size_t)L.P * 2 * L.bs * L.Hq * ((L.cap_sl + 3) / 4 * 4) * sizeof(float);
  return (rows + 1023) / 1024 * 1024;
}
size_t bwd_ds_bytes(const Layer& L, int64_t nblk) {
  return (size_t)dkdv::kDSBlock + (size_t)L.bs * L.hc * (size_t)nblk * 2 * dkdv::kDSBlock;
}


// dQ of ranks [r0, r0 + nr) from the stored dS blocks (R rows per tensor
// map, mk kv heads and mq query heads per map, as for the other passes).
static int launch_dq_stored(const Layer& L, const void* const* k, void* const* dq, const char* ds, const char* zero,
                            int r0, int nr, int64_t R, int mk, int mq, bool fused, cudaStream_t stream) {
  DqsParams d;
  for (int i = 0; i < nr; ++i) {
    const int r = r0 + i;
    if (!make_tmap_bf16_4d(&d.tk[i], k[r], 128, mk, L.bs, R, 64, 128) ||
        !make_tmap_bf16_4d(&d.tq[i], dq[r], 128, mq, L.bs, R, 64, 128))
      return ULYSSES_ERR_CUDA;
  }
  d.range = L.d_qp_range;
  d.order = L.d_qp_order;
  d.kv_range = L.d_kvp_range;
  d.ds_base = L.d_ds_base;
  d.ds = ds;
  d.zero = zero;
  d.ds_nblk = L.ds_nblk;
  d.status = L.d_status;
  d.timeout = L.timeout_cycles;
  d.bs = (int)L.bs;
  d.Hq = L.Hq;
  d.Hk = L.Hk;
  d.group = L.Hq / L.Hk;
  d.nranks = nr;
  d.fused = fused ? 1 : 0;
  d.n = (int)L.n();
  d.scale = (float)(1.0 / sqrt((double)L.hs));
  const long long pairs = (long long)((L.sl + 255) / 256) * nr * L.bs * L.Hq;
  if (2 * pairs > 0x7fffffffLL) return ULYSSES_ERR_UNSUPPORTED;
  Timed t(L.timing, ULYSSES_KERNEL_BWD_DQ, stream);
  attn_bwd_dq_stored_kernel<<<(unsigned)(2 * pairs), dqs::kThreads, dqs::kSmem, stream>>>(d);
  t.done();
  count_launches(1);
  return ULYSSES_OK;
}

int launch_attn_bwd_sm103(const Layer& L, const void* const* q, const void* const* k, const void* const* v,
                          const void* const* o, const void* const* dO, const float* const* lse, void* const* dq,
                          void* const* dk, void* const* dv, void* workspace, cudaStream_t stream, bool fused,
                          bool store_ds) {
  if (fused && !fused_supported(L)) return ULYSSES_ERR_UNSUPPORTED;
  static PerDeviceOnce attrs;
  const int ast = attrs.run([] {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dkdv::Layout<false>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)dkdv::Layout<true>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dqk::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dq_stored_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)dqs::kSmem);
    return e;
  });
  if (ast != ULYSSES_OK) return ast;
  // Workspace: per rank two row planes, -LSE*log2(e) then D, each
  // [bs*Hq][pitch] fp32 with the pitch a multiple of 16 bytes (a TMA stride).
  float* ws = reinterpret_cast<float*>(workspace);
  const long long pitch = bwd_row_pitch(L);
  const long long nrows = (long long)L.bs * L.Hq;
  const long long per_rank = 2 * nrows * pitch;
  // Stored dS: the zero block, then the blocks of every (rank, batch, head).
  store_ds = store_ds && L.ds_fits();
  char* ds_zero = store_ds ? reinterpret_cast<char*>(workspace) + bwd_ds_offset(L) : nullptr;
  char* ds = store_ds ? ds_zero + dkdv::kDSBlock : nullptr;
  const size_t ds_per_rank = (size_t)L.bs * L.Hq * (size_t)L.ds_nblk * 2 * dkdv::kDSBlock;

  // 1. The row planes.
  {
    PrepParams a;
    for (int r = 0; r < L.P; ++r) {
      a.o[r] = reinterpret_cast<const __nv_bfloat16*>(o[r]);
      a.dO[r] = reinterpret_cast<const __nv_bfloat16*>(dO[r]);
      a.lse[r] = lse[r];
      a.rows[r] = ws + per_rank * r;
    }
    a.P = L.P;
    a.sl = (int)L.sl;
    a.bs = (int)L.bs;
    a.Hq = L.Hq;
    a.pitch = (int)pitch;
    a.fused = fused ? 1 : 0;
    a.n = (int)L.n();
    a.zero = reinterpret_cast<uint4*>(ds_zero);
    Timed t(L.timing, ULYSSES_KERNEL_BWD_PREP, stream);
    const long long prep_rows = (long long)L.sl * L.bs * L.Hq;  // rows of each O / dO buffer
    const dim3 grid((unsigned)((prep_rows + kPrepRows - 1) / kPrepRows), (unsigned)L.P);
    attn_bwd_prep_kernel<<<grid, 256, 0, stream>>>(a);
    t.done();
    count_launches(1);
  }
  PairParams prm;
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
  prm.pitch = (int)pitch;
  prm.fused = fused ? 1 : 0;
  prm.n = (int)L.n();
  prm.skip_q_loads = 0;
  prm.ds_base = L.d_ds_base;
  prm.ds_nblk = L.ds_nblk;
  const bool inject = L.inject_fault == 2;
  if (inject) L.inject_fault = 0;
  prm.scale = (float)(1.0 / sqrt((double)L.hs));
  prm.scale_log2 = (float)(1.4426950408889634 / sqrt((double)L.hs));
  const int n_pair = (int)((L.sl + 255) / 256);
  // Fused: one launch covers all P ranks, and map i is sequence shard i,
  // [n][bs][H][hs] with every head. Otherwise map i is head shard r0 + i.
  const int64_t R = fused ? L.n() : L.sl;
  const int mq = fused ? L.hc : L.Hq, mk = fused ? L.hkv : L.Hk;
  for (int pass = 0; pass < 2; ++pass) {  // 2. dK, dV   3. dQ
    prm.range = pass == 0 ? L.d_kvp_range : L.d_qp_range;
    prm.order = pass == 0 ? L.d_kvp_order : L.d_qp_order;
    for (int r0 = 0; r0 < L.P; r0 += kRanksPerLaunch) {
      const int nr = std::min(kRanksPerLaunch, L.P - r0);
      if (pass == 1 && store_ds) {
        const int st = launch_dq_stored(L, k, dq, ds + ds_per_rank * r0, ds_zero, r0, nr, R, mk, mq, fused, stream);
        if (st != ULYSSES_OK) return st;
        continue;
      }
      prm.nranks = nr;
      prm.ds = (pass == 0 && store_ds) ? ds + ds_per_rank * r0 : nullptr;
      prm.skip_q_loads = (inject && pass == 0) ? 1 : 0;
      for (int i = 0; i < nr; ++i) {
        const int r = r0 + i;
        bool ok;
        if (pass == 0)
          ok = make_tmap_bf16_4d(&prm.ta[i], k[r], 128, mk, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.tb[i], v[r], 128, mk, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.tc[i], q[r], 128, mq, L.bs, R, 64, 64) &&
               make_tmap_bf16_4d(&prm.td[i], dO[r], 128, mq, L.bs, R, 64, 64) &&
               make_tmap_bf16_4d(&prm.te[i], q[r], 128, mq, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.tf[i], dO[r], 128, mq, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.tg[i], dk[r], 128, mk, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.th[i], dv[r], 128, mk, L.bs, R, 64, 128) &&
               make_tmap_f32_rows(&prm.tr[i], ws + per_rank * r, (uint64_t)L.sl, (uint64_t)nrows,
                                  (uint64_t)pitch);
        else
          ok = make_tmap_bf16_4d(&prm.ta[i], q[r], 128, mq, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.tb[i], dO[r], 128, mq, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.tc[i], k[r], 128, mk, L.bs, R, 64, 64) &&
               make_tmap_bf16_4d(&prm.td[i], v[r], 128, mk, L.bs, R, 64, 64) &&
               make_tmap_bf16_4d(&prm.te[i], k[r], 128, mk, L.bs, R, 64, 128) &&
               make_tmap_bf16_4d(&prm.tf[i], dq[r], 128, mq, L.bs, R, 64, 128);
        if (!ok) return ULYSSES_ERR_CUDA;
        prm.rows[i] = ws + per_rank * r;
      }
      const long long pairs = (long long)n_pair * nr * L.bs * (pass == 0 ? L.Hk : L.Hq);
      if (2 * pairs > 0x7fffffffLL) return ULYSSES_ERR_UNSUPPORTED;
      Timed t(L.timing, pass == 0 ? ULYSSES_KERNEL_BWD_DKDV : ULYSSES_KERNEL_BWD_DQ, stream);
      if (pass == 0 && store_ds)
        attn_bwd_dkdv_kernel<true><<<(unsigned)(2 * pairs), kThreads, dkdv::Layout<true>::kSmem, stream>>>(prm);
      else if (pass == 0)
        attn_bwd_dkdv_kernel<false><<<(unsigned)(2 * pairs), kThreads, dkdv::Layout<false>::kSmem, stream>>>(prm);
      else
        attn_bwd_dq_kernel<<<(unsigned)(2 * pairs), kThreads, dqk::kSmem, stream>>>(prm);
      t.done();
      count_launches(1);
    }
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace uly
