// attn_fwd_sm103.cu — causal / per-document attention forward on the tcgen05 tensor cores.
//
// The computation is step 4 of the HF blog "Ulysses Sequence Parallelism:
// Training with Million-Token Contexts": standard attention for each head a
// rank holds, over the full sequence. Per head, with s = 1/sqrt(hs):
//   S = s Q K^T (masked),  O = softmax(S) V,  LSE = ln sum exp(S)
// The mask follows the position ids of the ALST guide (sections 2.1, 2.2):
// causal, and no key visible across a document boundary.
//
// Design (bf16 in, fp32 accumulate, head size 128):
//  * A cluster of two CTAs runs M=256 UMMAs (tcgen05 .cta_group::2): the
//    even CTA owns query rows [256m, 256m+128), the odd one the next 128.
//    Each CTA holds two query tiles, of two query heads of the same GQA
//    group at the same rows: every K/V tile in shared memory feeds both.
//  * Per 128-key tile each CTA loads half of K (its 64 keys x 128, the N
//    half of the B operand of S = Q K^T) and half of V (128 keys x its 64
//    head columns, the N half of the B operand of O += P V). The even CTA's
//    UMMA issuer drives both CTAs' tensor cores; the odd CTA forwards its
//    load completions to the even CTA's barriers.
//  * Warp roles: warps 0-3 and 4-7 are the softmax warpgroups of tile 0 and
//    tile 1 (one query row per thread, which is one TMEM lane); warp 8 issues
//    the TMA loads; warp 9 allocates tensor memory (both CTAs) and, in the
//    even CTA, issues the UMMAs; warp 10 of the odd CTA forwards. The block
//    launches with 168 registers per thread; the third warpgroup gives up
//    112 of them (down to 56) and the softmax warpgroups take them (up to
//    224): 2*128*224 + 128*56 = 384*168.
//  * Tensor memory (512 columns): S of tile t at columns [128t, 128t+128),
//    overwritten in place by P (bf16, 64 columns); O of tile t at
//    [256+128t, 384+128t). P feeds O += P V straight from tensor memory.
//  * The two tiles ping-pong: while one warpgroup exponentiates its S, the
//    tensor cores run the other tile's P V and Q K^T.
//  * Online softmax in the log2 domain. O is rescaled only when a row's max
//    grows by more than 8 (a factor 256), so the rescale is rare. The final
//    O = sum p v / sum p is exact whatever max was used. The per-element
//    arithmetic uses packed fp32 pairs, which leave the tensor pipe's rate
//    alone.
//  * Key tiles outside the visible range of the 256 rows are never loaded
//    (causal and per-document block skipping). The host orders the row
//    blocks by their number of key tiles, most first.
//  * Every mbarrier wait is bounded. A wait that runs out sets the handle's
//    status word, and the kernel winds down without touching more data.
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
constexpr int kRegsSoftmax = 224;
constexpr int kRegsOther = 56;
constexpr int kRegsLaunch = (65536 / kThreads) / 8 * 8;  // registers per thread at launch
static_assert(kRegsSoftmax >= kRegsLaunch && kRegsOther <= kRegsLaunch, "register split directions");
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kThreads * kRegsLaunch,
              "register split must add up to the launch budget");
constexpr int NS = 4;                              // K/V pipeline stages
constexpr uint32_t kTile = 128 * 128 * 2;          // one 128x128 bf16 tile: 32 KB
constexpr uint32_t kHalf = kTile / 2;              // 16 KB
constexpr uint32_t kOffQ = 0;                      // 2 query tiles
constexpr uint32_t kOffStage = 2 * kTile;          // NS stages: K half (16 KB), then V half (16 KB)
constexpr uint32_t kStage = 2 * kHalf;
constexpr uint32_t kOffBar = kOffStage + NS * kStage;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack

static_assert(kMaxFusedP <= kRanksPerLaunch, "a fused launch holds one tensor map per sequence shard");

// Tensor maps: one per rank of the launch (head shards), or one per sequence
// shard (fused; see locate_tile).
struct FwdParams {
  CUtensorMap tq[kRanksPerLaunch];   // Q, boxes of 64 columns x 128 rows
  CUtensorMap tk[kRanksPerLaunch];   // K, boxes of 64 columns x 64 rows
  CUtensorMap tv[kRanksPerLaunch];   // V, boxes of 64 columns x 128 rows
  CUtensorMap to[kRanksPerLaunch];   // O (store), boxes of 64 columns x 128 rows
  float* lse[kRanksPerLaunch];       // per rank of the launch
  const int2* kv_range;   // per 256-row block: first and last key tile (inclusive)
  const int* m_order;     // row blocks, most key tiles first
  const int32_t* doc_offsets;
  unsigned* status;
  long long timeout;      // clock cycles per wait
  int ndoc, sl, bs, Hq, Hk, group, npairs, nranks, causal;
  int fused;              // operands are sequence shards of n tokens (nranks = P)
  int n;
  int skip_kv_loads;      // test hook: the producer issues no K/V loads
  float scale_log2;
};

// Barrier indices.
enum {
  B_QFULL = 0,               // Q landed (even CTA: + the odd CTA's forward)
  B_KVFULL = 1,              // NS: K/V halves landed (even CTA: + forward)
  B_KVEMPTY = B_KVFULL + NS, // NS: stage consumed (1 softmax thread, this CTA)
  B_SFULL = B_KVEMPTY + NS,  // 2: S of tile t ready (commit, both)
  B_PFULL = B_SFULL + 2,     // 2: even CTA: P of tile t written in both CTAs (8 warps)
  B_OFINAL = B_PFULL + 2,    // 2: every UMMA of tile t done (commit, both)
  B_OSTAGE = B_OFINAL + 2,   // 2: O of tile t staged (128 threads)
  B_DRAIN = B_OSTAGE + 2,
  B_COUNT
};
static_assert(8 * B_COUNT + 4 <= 256, "barrier area");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_sm103_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ0 = sb + kOffQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();

  // Pair work item: (256-row block, rank, batch, kv head, pair of query heads).
  const int pair = blockIdx.x >> 1;
  const int units = p.nranks * p.bs * p.Hk * p.npairs;
  const int mp = p.m_order[pair / units];
  int rest = pair % units;
  const int hpair = rest % p.npairs;
  rest /= p.npairs;
  const int hk = rest % p.Hk;
  rest /= p.Hk;
  const int b = rest % p.bs;
  const int rl = rest / p.bs;
  const int hq0 = hk * p.group + 2 * hpair;
  const int ntile = (2 * hpair + 1 < p.group) ? 2 : 1;
  const int2 kr = p.kv_range[mp];
  const int n_kv = kr.y - kr.x + 1;
  const int q0 = mp * 256 + 128 * (int)crank;  // this CTA's first query row

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_QFULL || (i >= B_KVFULL && i < B_KVFULL + NS)) cnt = crank == 0 ? 2 : 1;
      if (i == B_PFULL || i == B_PFULL + 1) cnt = 8;
      if (i == B_OSTAGE || i == B_OSTAGE + 1) cnt = 128;
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
  cluster_sync();  // barriers of both CTAs exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = p.timeout;

  if (warp >= 8) {
    regs_dec<kRegsOther>();
    if (warp == 8) {
      // ----------------------------------------------------------------- TMA producer
      if (lane == 0) {
        bool ok = true;
        int last[NS];  // last phase armed on each full barrier (-1: none)
        for (int i = 0; i < NS; ++i) last[i] = -1;
        mbar_expect_tx(bar(B_QFULL), ntile * kTile);
        for (int t = 0; t < ntile; ++t) {
          const uint32_t dst = sQ0 + t * kTile;
          const TileLoc lq = locate_tile(p.fused, p.n, p.nranks, rl, p.Hq, hq0 + t, q0);
          tma_load_4d(dst, &p.tq[lq.map], bar(B_QFULL), 0, lq.head, b, lq.row);
          tma_load_4d(dst + kHalf, &p.tq[lq.map], bar(B_QFULL), 64, lq.head, b, lq.row);
        }
        for (int jj = 0; jj < (p.skip_kv_loads ? 0 : n_kv); ++jj) {
          const int st = jj % NS, u = jj / NS;
          const int k0 = (kr.x + jj) * 128;
          if (!mbar_wait(bar(B_KVEMPTY + st), (u & 1) ^ 1, lim)) { ok = false; break; }
          const uint32_t sk = sb + kOffStage + st * kStage;
          mbar_expect_tx(bar(B_KVFULL + st), kStage);
          // the tile's 128 keys are in one shard
          const TileLoc l = locate_tile(p.fused, p.n, p.nranks, rl, p.Hk, hk, k0);
          // K rows [k0 + 64c, +64) (the N half of B for S = Q K^T), K-major in two 64-column boxes
          tma_load_4d(sk, &p.tk[l.map], bar(B_KVFULL + st), 0, l.head, b, l.row + 64 * (int)crank);
          tma_load_4d(sk + kHalf / 2, &p.tk[l.map], bar(B_KVFULL + st), 64, l.head, b, l.row + 64 * (int)crank);
          // V columns [64c, 64c+64) of all 128 key rows (the N half of B for O += P V), MN-major
          tma_load_4d(sk + kHalf, &p.tv[l.map], bar(B_KVFULL + st), 64 * (int)crank, l.head, b, l.row);
          last[st] = u;
        }
        if (!ok) atomicOr(p.status, STATUS_TIMEOUT);
        // Let every copy this thread started land before the CTA can exit.
        mbar_wait(bar(B_QFULL), 0, lim);
        for (int i = 0; i < NS; ++i)
          if (last[i] >= 0) mbar_wait(bar(B_KVFULL + i), last[i] & 1, lim);
      }
      __syncwarp();
    } else if (warp == 9 && crank == 0) {
      // ----------------------------------------------------------------- UMMA issuer (even CTA)
      if (lane == 0) {
        constexpr uint32_t idesc_s = idesc_bf16_f32(256, 128, 0, 0);  // Q (K-major) x K (K-major)
        constexpr uint32_t idesc_o = idesc_bf16_f32(256, 128, 0, 1);  // P (tmem) x V (MN-major)
        // Descriptors are formed once per tile and stepped by constants, so
        // that each UMMA costs the issuing thread one add.
        auto issue_s = [&](int t, int st) {
          const uint64_t dq = sdesc_sw128(sQ0 + t * kTile, 0, 1024);
          const uint64_t dk = sdesc_sw128(sb + kOffStage + st * kStage, 0, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma2_ss(tmem + t * 128, sdesc_add(dq, (kk >> 2) * kHalf + (kk & 3) * 32),
                     sdesc_add(dk, (kk >> 2) * (kHalf / 2) + (kk & 3) * 32), idesc_s, kk > 0);
        };
        auto issue_pv = [&](int t, int st, bool acc) {
          const uint64_t dv = sdesc_sw128(sb + kOffStage + st * kStage + kHalf, kHalf, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma2_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, sdesc_add(dv, kk * 2048), idesc_o,
                     (acc || kk > 0) ? 1u : 0u);
        };
        bool ok = mbar_wait(bar(B_QFULL), 0, lim) && mbar_wait(bar(B_KVFULL), 0, lim);
        if (ok) {
          tc_fence_after();
          for (int t = 0; t < ntile; ++t) {
            issue_s(t, 0);
            umma2_commit_both(bar(B_SFULL + t));
          }
        }
        for (int jj = 0; jj < n_kv && ok; ++jj) {
          const int st = jj % NS;
          const bool next = jj + 1 < n_kv;
          const int st1 = (jj + 1) % NS, u1 = (jj + 1) / NS;
          for (int t = 0; t < ntile; ++t) {
            if (!mbar_wait(bar(B_PFULL + t), jj & 1, lim)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, st, jj > 0);
            if (next) {
              if (t == 0) {
                if (!mbar_wait(bar(B_KVFULL + st1), u1 & 1, lim)) { ok = false; break; }
                tc_fence_after();
              }
              issue_s(t, st1);  // over P of this tile: after the P V above has read it
              umma2_commit_both(bar(B_SFULL + t));
            }
          }
          if (!ok) break;
        }
        if (ok) {
          for (int t = 0; t < ntile; ++t) umma2_commit_both(bar(B_OFINAL + t));
        } else {
          atomicOr(p.status, STATUS_TIMEOUT);
        }
        // Every UMMA issued so far completes before the tensor memory is freed.
        umma2_commit_both(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, lim);
      }
      __syncwarp();
    } else if (warp == 10 && crank == 1) {
      // ----------------------------------------------------------------- forwarder (odd CTA)
      // The even CTA's UMMAs read this CTA's shared memory: tell it when the
      // loads have landed.
      if (lane == 0) {
        bool ok = mbar_wait(bar(B_QFULL), 0, lim);
        if (ok) mbar_arrive_cluster(mapa(bar(B_QFULL), 0));
        for (int jj = 0; jj < (p.skip_kv_loads ? 0 : n_kv) && ok; ++jj) {
          const int st = jj % NS, u = jj / NS;
          ok = mbar_wait(bar(B_KVFULL + st), u & 1, lim);
          if (ok) mbar_arrive_cluster(mapa(bar(B_KVFULL + st), 0));
        }
        if (!ok) atomicOr(p.status, STATUS_TIMEOUT);
      }
      __syncwarp();
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ----------------------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;
    if (t < ntile) {
      const int rq = (warp & 3) * 32 + lane;  // row within the tile = TMEM lane
      const int row = q0 + rq;
      const int hq = hq0 + t;
      int lo = 0, hi = -1;                      // visible keys [lo, hi] of this row
      if (row < p.sl) {
        const int d = doc_of(p.doc_offsets, p.ndoc, row);
        lo = p.doc_offsets[d];
        hi = p.causal ? row : p.doc_offsets[d + 1] - 1;
      }
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t t_s = tmem + lane_base + t * 128;
      const uint32_t t_o = tmem + lane_base + 256 + t * 128;
      const float sl2 = p.scale_log2;
      const uint64_t sc2 = f2(sl2, sl2);
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int jj = 0; jj < n_kv; ++jj) {
        ok = warp_wait(bar(B_SFULL + t), jj & 1, lim);
        if (!ok) break;
        tc_fence_after();
        // S of the last tile for key tile jj is the last UMMA issued for key
        // tile jj-1: once it has completed, that tile's K/V stage is free.
        if (t == ntile - 1 && rq == 0 && jj > 0) mbar_arrive(bar(B_KVEMPTY + (jj - 1) % NS));
        __syncwarp();
        uint32_t s[128];
        tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
        tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        tmem_ld_wait(s);
        const int kb = (kr.x + jj) * 128;
        if (!(lo <= kb && kb + 127 <= hi)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int key = kb + c;
            if (key < lo || key > hi) s[c] = __float_as_uint(-INFINITY);
          }
        }
        // row max: four independent chains of three-input maxes
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; c += 8)
#pragma unroll
          for (int j = 0; j < 4; ++j) mq[j] = fmax3(mq[j], __uint_as_float(s[c + 2 * j]), __uint_as_float(s[c + 2 * j + 1]));
        const float mx = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
        const float mx2 = mx * sl2;
        const bool need = mx2 > m_used + 8.0f;
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m_used - mx2);
          m_used = mx2;
          l *= alpha;
        }
        if (jj > 0 && __any_sync(0xffffffffu, need)) {
          // O holds the sum over earlier key tiles (their P V completed before
          // this tile's S was committed); scale it to the new max.
          const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            tmem_ld32(t_o + 32 * q, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              float lo2, hi2;
              f2_split(f2_mul(f2_bits(o[2 * c], o[2 * c + 1]), a2), lo2, hi2);
              o[2 * c] = __float_as_uint(lo2);
              o[2 * c + 1] = __float_as_uint(hi2);
            }
            tmem_st32(t_o + 32 * q, o);
          }
          tmem_st_wait();
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        // P = 2^(S * scale*log2(e) - m), two keys per packed op; four partial row sums
        const uint64_t nm2 = f2(-msub, -msub);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const uint64_t pp = f2_ex2(f2_fma(f2_bits(s[2 * c], s[2 * c + 1]), sc2, nm2));
          sum2[c & 3] = f2_add(sum2[c & 3], pp);
          s[c] = f2_pack_bf16(pp);
        }
        float s0, s1;
        f2_split(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), s0, s1);
        l += s0 + s1;
        tmem_st32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_st_wait();
        tc_fence_before();
        warp_arrive_leader(bar(B_PFULL + t), crank);
      }
      if (ok) ok = warp_wait(bar(B_OFINAL + t), 0, lim);
      if (ok) {
        tc_fence_after();
        // Normalise O and stage it, 128-byte swizzled, in this tile's Q buffer
        // (free: every UMMA has completed), then one TMA store per half.
        const float inv = 1.f / l;
        const uint64_t inv2 = f2(inv, inv);
        const uint32_t stage = sQ0 + t * kTile;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[32];
          tmem_ld32(t_o + 32 * q, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = f2_pack_bf16(f2_mul(f2_bits(o[c4 * 8 + 2 * e], o[c4 * 8 + 2 * e + 1]), inv2));
            const int chunk = q * 4 + c4;  // 16-byte chunk of the 256-byte row
            const uint32_t addr = stage + (chunk >> 3) * kHalf + sw128_offset(rq, chunk & 7);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_OSTAGE + t));
        if (rq == 0) {
          if (mbar_wait(bar(B_OSTAGE + t), 0, lim)) {
            const TileLoc lo_ = locate_tile(p.fused, p.n, p.nranks, rl, p.Hq, hq, q0);
            tma_store_4d(&p.to[lo_.map], stage, 0, lo_.head, b, lo_.row);
            tma_store_4d(&p.to[lo_.map], stage + kHalf, 64, lo_.head, b, lo_.row);
            bulk_commit();
            bulk_wait_read_all();  // the stores have read shared memory; their global writes complete before the grid does
          } else {
            atomicOr(p.status, STATUS_TIMEOUT);
          }
        }
        if (row < p.sl) p.lse[rl][((size_t)b * p.Hq + hq) * p.sl + row] = (m_used + log2f(l)) * 0.69314718055994531f;
      } else if (lane == 0) {
        atomicOr(p.status, STATUS_TIMEOUT);
      }
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

}  // namespace

bool fwd_sm103_supported(const Layer& L) { return L.dtype == ULYSSES_BF16 && L.hs == 128; }

bool fused_supported(const Layer& L) {
  return fwd_sm103_supported(L) && L.P <= kMaxFusedP && L.n() % 128 == 0 && L.hkv % L.P == 0;
}

int launch_attn_fwd_sm103(Layer& L, const void* const* q, const void* const* k, const void* const* v,
                          void* const* o, float* const* lse, cudaStream_t stream, bool fused) {
  static PerDeviceOnce attrs;
  const int st = attrs.run([] {
    return cudaFuncSetAttribute(attn_fwd_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  });
  if (st != ULYSSES_OK) return st;
  const int n_pair = (int)((L.sl + 255) / 256);
  const int group = L.Hq / L.Hk;
  FwdParams prm;
  prm.kv_range = L.d_qp_range;
  prm.m_order = L.d_qp_order;
  prm.doc_offsets = L.d_doc_offsets;
  prm.status = L.d_status;
  prm.timeout = L.timeout_cycles;
  prm.ndoc = L.ndoc;
  prm.sl = (int)L.sl;
  prm.bs = (int)L.bs;
  prm.Hq = L.Hq;
  prm.Hk = L.Hk;
  prm.group = group;
  prm.npairs = (group + 1) / 2;
  prm.causal = L.causal;
  prm.skip_kv_loads = L.inject_fault == 1 ? 1 : 0;
  if (L.inject_fault == 1) L.inject_fault = 0;
  prm.scale_log2 = (float)(1.4426950408889634 / sqrt((double)L.hs));
  prm.fused = fused ? 1 : 0;
  prm.n = (int)L.n();
  if (fused && !fused_supported(L)) return ULYSSES_ERR_UNSUPPORTED;
  // Fused: one launch covers all P ranks, and map i is sequence shard i,
  // [n][bs][H][hs] with every head. Otherwise map i is head shard r0 + i.
  const int64_t rows = fused ? L.n() : L.sl;
  const int mq = fused ? L.hc : L.Hq, mk = fused ? L.hkv : L.Hk;
  for (int r0 = 0; r0 < L.P; r0 += kRanksPerLaunch) {
    const int nr = std::min(kRanksPerLaunch, L.P - r0);
    prm.nranks = nr;
    for (int i = 0; i < nr; ++i) {
      const int r = r0 + i;
      bool ok = make_tmap_bf16_4d(&prm.tq[i], q[r], 128, mq, L.bs, rows, 64, 128) &&
                make_tmap_bf16_4d(&prm.tk[i], k[r], 128, mk, L.bs, rows, 64, 64) &&
                make_tmap_bf16_4d(&prm.tv[i], v[r], 128, mk, L.bs, rows, 64, 128) &&
                make_tmap_bf16_4d(&prm.to[i], o[r], 128, mq, L.bs, rows, 64, 128);
      if (!ok) return ULYSSES_ERR_CUDA;
      prm.lse[i] = lse[r];
    }
    const long long pairs = (long long)n_pair * nr * L.bs * L.Hk * prm.npairs;
    if (2 * pairs > 0x7fffffffLL) return ULYSSES_ERR_UNSUPPORTED;
    Timed t(L.timing, ULYSSES_KERNEL_ATTN_FWD, stream);
    attn_fwd_sm103_kernel<<<(unsigned)(2 * pairs), kThreads, kSmemBytes, stream>>>(prm);
    t.done();
    count_launches(1);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return ULYSSES_ERR_CUDA;
  }
  return ULYSSES_OK;
}

}  // namespace uly
