// MoDA forward for d = 64: two query tiles per CTA in ping-pong (sm_103a).
//
// Same method and tiling as the d = 128 kernel (fwd_tc.cu): G-stacked
// 128-row query tiles, 128-key sequence blocks under the grouped causal mask,
// depth blocks under the block-diagonal mask, one online softmax per row.
// At d = 64 a block costs the tensor core half as much while its softmax costs
// the same, so one tile per CTA leaves the tensor core idle most of the time.
// Here a CTA owns two adjacent tiles A and B of one KV head (positions
// [p0, p0+P) and [p0+P, p0+2P), P = 128/G): they read the same K/V blocks,
// which are staged once, and each tile has its own softmax warpgroup and its
// own MMA issuer, so one tile's softmax overlaps the other tile's MMAs.
//
// Persistent CTAs, as at d = 128: one CTA per SM takes pairs from a queue in
// global memory (KV-head-major, longest pair first within a head). Stage and
// barrier phases run on across pairs, so the next pair's K/V blocks load
// while the current one finishes and a pair costs no launch, prologue or
// pipeline drain; the next pair's Q lands once every S product of the current
// pair has read Q, and its first S products run during the current pair's
// epilogue.
//
// Roles (12 warps): warp 0 takes the pairs from the queue and passes them on
// through a ring in shared memory, and loads the K blocks; warp 2 loads Q_A,
// Q_B and the V blocks; warp 1 issues tile A's MMAs, warp 3 tile B's; warps 4-7 are
// tile A's softmax and epilogue, warps 8-11 tile B's (thread = row = TMEM
// lane). TMEM: S_A [0,128), S_B [128,256), O_A [256,320), O_B [320,384),
// P_A [384,448), P_B [448,512). Each issuer runs its S stream one used block
// ahead of its P.V stream: S_X(j+1) once the softmax holds S_X(j) in
// registers, P_X(j).V(j) once P_X(j) is stored (the S cursor runs at most
// two blocks ahead of the P.V cursor).
// Depth blocks belong to one tile: as in the d = 128 kernel, each of its
// softmax warps owns one 32-row word of the block, filled with the next packed
// depth rows of the warp's own positions (or, from layer-major depth tensors,
// gathered by a 4-D copy box of its PW positions x 32/PW slots). A tile's
// depth blocks are its own
// (A's first, then B's in the pair's schedule); the last sequence block may be
// used by both tiles. Every K/V stage is
// released by two arrivals per block, one per tile: the MMA commit of a tile
// that used the block, or a plain arrive of one that did not, made only
// after the block's full barrier, so an early arrival never completes the
// previous block's phase.
// The softmax warpgroups get 216 registers each and the TMA/MMA warpgroup 64
// (128 x 64 + 256 x 216 = 63488, within the launch allocation of 384 x 168).
// Every wait is bounded (2 s); on expiry the CTA drains, frees TMEM and
// latches MODA_ERR_TIMEOUT.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "softmax_block.cuh"
#include "tensor_map.h"

namespace moda {
namespace {

using namespace sm103;

constexpr int D = 64;
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 384;
constexpr int kNS = 6;  // K and V stages
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kSumBound = 256.0f;         // 2^kRescaleThreshold

constexpr int kTile = 128 * D * 2;  // one 128-row, 64-column box (16 KB)
constexpr int kOffQ = 0;            // Q_A, Q_B
constexpr int kOffK = 2 * kTile;
constexpr int kOffV = kOffK + kNS * kTile;
constexpr int kOffBar = kOffV + kNS * kTile;
constexpr int kSmemBytes = kOffBar + 512 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;

constexpr int kPairRing = 4;  // pair numbers in flight between roles
// arrivals that free a pair-ring entry: V producer, two MMA issuers, 8 softmax warps
constexpr int kPairReaders = 11;

struct alignas(8) PpBars {
  uint64_t q_full;  // Q_A, Q_B of the current pair landed
  uint64_t q_free;  // every S product of the previous pair completed (one commit per issuer)
  uint64_t k_full[kNS], k_empty[kNS];
  uint64_t v_full[kNS], v_empty[kNS];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];  // per tile
  uint64_t t_full[kPairRing], t_empty[kPairRing];
  uint64_t mma_done[2];
  int pair_ring[kPairRing];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PpBars) <= 512, "barrier block");

struct PpParams {
  int T, Hq, Hk, L, lgG, npairs, total;
  int depth_lm;  // depth K/V layer-major [L, T, Hk, d] (else packed [Hk, T, L, d])
  float scale_log2;
  __nv_bfloat16* o;
  int o_v8;  // o is 32-byte aligned: rows go out in 32-byte stores
  float* lse;
  unsigned int* err;
  unsigned int* queue;  // {next pair, CTAs finished}
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

// The pair's blocks in order: the n_depth depth blocks spread among the
// sequence blocks (Bresenham), and which tiles use each.
struct PairSched {
  int acc = 0, db = 0, sbk = 0;
  bool depth = false;
  int index = 0;
  __device__ void next(int n_depth, int nb) {
    acc += n_depth;
    depth = acc >= nb;
    if (depth) {
      acc -= nb;
      index = db++;
    } else {
      index = sbk++;
    }
  }
};

// Geometry of queue entry o: KV-head-major, longest pair first within a head
// (the CTAs at work share one or two heads' K/V in L2).
struct PairGeom {
  int hk;
  int P;        // positions per tile
  int p0;       // first position of tile A (tile B starts at p0 + P)
  int npos[2];  // positions of A and B (0: B absent)
  int nb_seq[2];
  int nd[2];    // depth blocks of A and B: ceil(min(npos, P/4) * L / 32)
  int n_depth, nb;
  int PW, RW;   // positions and packed depth rows per softmax warp
  int depth_row0;  // tile A's first packed depth row
  __device__ void set(int o, const PpParams& p) {
    const int pp = p.npairs - 1 - o % p.npairs;
    hk = o / p.npairs;
    P = BM >> p.lgG;
    p0 = pp * 2 * P;
    npos[0] = min(P, p.T - p0);
    npos[1] = p0 + P < p.T ? min(P, p.T - p0 - P) : 0;
    for (int x = 0; x < 2; ++x) nb_seq[x] = npos[x] ? (p0 + x * P + npos[x] - 1) / BN + 1 : 0;
    PW = P >> 2;
    RW = PW * p.L;
    // a word holds 32 rows: 32 consecutive packed rows, or (layer-major) PW
    // positions x 32/PW slots
    for (int x = 0; x < 2; ++x) nd[x] = npos[x] ? ((p.depth_lm ? PW : min(npos[x], PW)) * p.L + 31) / 32 : 0;
    n_depth = nd[0] + nd[1];
    nb = n_depth + max(nb_seq[0], nb_seq[1]);
    depth_row0 = (hk * p.T + p0) * p.L;
  }
  // the tile a depth block belongs to, and its index among that tile's
  __device__ int depth_tile(int index) const { return index < nd[0] ? 0 : 1; }
  __device__ int depth_index(int index) const { return index < nd[0] ? index : index - nd[0]; }
  __device__ bool uses(int x, const PairSched& s) const {
    if (npos[x] == 0) return false;
    if (!s.depth) return s.index < nb_seq[x];
    return depth_tile(s.index) == x;
  }
};

// The k-th pair of this CTA from the ring (-1: no more pairs); the reader
// frees the entry right away. False on a timeout.
__device__ __forceinline__ bool read_pair(PpBars* bars, int k, volatile int* abort, int* o, bool arrive) {
  const int s = k % kPairRing;
  if (!warp_wait(smem_u32(&bars->t_full[s]), (k / kPairRing) & 1, abort)) return false;
  *o = *reinterpret_cast<volatile int*>(&bars->pair_ring[s]);
  __syncwarp();
  if (arrive) mbar_arrive(smem_u32(&bars->t_empty[s]));
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
moda_fwd_pp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKd,
                   const __grid_constant__ CUtensorMap tmVd, const PpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  PpBars* bars = reinterpret_cast<PpBars*>(smem + kOffBar);
  const uint32_t sQ = smem_u32(smem + kOffQ), sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = 1 << p.lgG;

  if (tid == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_free), 2);  // one commit per MMA issuer and pair
    for (int s = 0; s < kNS; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->k_empty[s]), 2);  // one arrival per tile and block
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->v_empty[s]), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&bars->s_full[x]), 1);
      mbar_init(smem_u32(&bars->s_free[x]), 128);
      mbar_init(smem_u32(&bars->p_full[x]), 128);
      mbar_init(smem_u32(&bars->pv_done[x]), 1);
      mbar_init(smem_u32(&bars->mma_done[x]), 1);
    }
    for (int s = 0; s < kPairRing; ++s) {
      mbar_init(smem_u32(&bars->t_full[s]), 1);
      mbar_init(smem_u32(&bars->t_empty[s]), kPairReaders);
    }
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (p.L) {
      tma_prefetch_desc(&tmKd);
      tma_prefetch_desc(&tmVd);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;\n" ::: "memory");
    if (warp == 0 || warp == 2) {
      // ---------------------------------------------------- TMA producers
      // Stages and phases follow the CTA's running block count gb across
      // pairs. Warp 0 takes the pairs from the queue and passes them on; warp
      // 2 loads each pair's Q once both issuers' S products of the previous
      // pair have completed (they read Q from shared memory).
      const bool leader = elect_one();
      const bool is_k = warp == 0;
      const uint32_t sbase = is_k ? sK : sV;
      const CUtensorMap* seq_map = is_k ? &tmK : &tmV;
      const CUtensorMap* dep_map = is_k ? &tmKd : &tmVd;
      uint64_t* full = is_k ? bars->k_full : bars->v_full;
      uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
      const uint64_t pol_once = l2_policy_evict_first();
      int gb = 0;  // blocks issued so far, over all pairs
      int nq = 0;  // Q loads issued
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int o;
        if (is_k) {
          const int s = k % kPairRing;
          if (!warp_wait(smem_u32(&bars->t_empty[s]), ((k / kPairRing) & 1) ^ 1, abort)) break;
          if (leader) {
            const unsigned int t = atomicAdd(p.queue, 1u);
            o = t < (unsigned int)p.total ? (int)t : -1;
            *reinterpret_cast<volatile int*>(&bars->pair_ring[s]) = o;
            mbar_arrive(smem_u32(&bars->t_full[s]));
          }
          o = __shfl_sync(0xffffffffu, o, __ffs(__ballot_sync(0xffffffffu, leader)) - 1);
        } else if (!read_pair(bars, k, abort, &o, leader)) {
          break;
        }
        if (o < 0) break;
        PairGeom g;
        g.set(o, p);
        if (!is_k) {
          if (k > 0 && !warp_wait(smem_u32(&bars->q_free), (k - 1) & 1, abort)) break;
          if (leader) {
            const uint32_t qb = smem_u32(&bars->q_full);
            mbar_arrive_expect_tx(qb, (g.npos[1] ? 2 : 1) * kTile);
            tma_load_3d_hint(sQ, &tmQ, qb, 0, g.hk * G, g.p0, pol_once);
            if (g.npos[1]) tma_load_3d_hint(sQ + kTile, &tmQ, qb, 0, g.hk * G, g.p0 + g.P, pol_once);
          }
          ++nq;
        }
        PairSched sch;
        for (int j = 0; j < g.nb; ++j, ++gb) {
          sch.next(g.n_depth, g.nb);
          const int s = gb % kNS;
          if (!warp_wait(smem_u32(&empty[s]), ((gb / kNS) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          if (leader) {
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, kTile);
            const uint32_t dst = sbase + s * kTile;
            if (sch.depth) {
              // four 32-row words: rows [32w, 32w+32) of the stage hold softmax
              // warp w's next 32 packed depth rows of the block's tile
              const int x = g.depth_tile(sch.index);
              if (p.depth_lm) {
                // layer-major: the copy gathers slots [SP*i, SP*i + SP) of warp
                // w's PW positions, row l_local*PW + t_local (SP = 32/PW)
                const int SP = 32 / g.PW;
                for (int w = 0; w < 4; ++w)
                  tma_load_4d_hint(dst + w * 32 * 128, dep_map, fb, 0, g.hk, g.p0 + x * g.P + w * g.PW,
                                   g.depth_index(sch.index) * SP, pol_once);
              } else {
                const int r0 = g.depth_row0 + x * g.P * p.L + g.depth_index(sch.index) * 32;
                for (int w = 0; w < 4; ++w)
                  tma_load_2d_hint(dst + w * 32 * 128, dep_map, fb, 0, r0 + w * g.RW, pol_once);
              }
            } else
              tma_load_3d(dst, seq_map, fb, 0, g.hk, sch.index * BN);
          }
          __syncwarp();
        }
      }
      if (leader) {  // every copy this warp issued lands before shared memory is released
        int never = 0;
        for (int j = max(0, gb - kNS); j < gb; ++j)
          mbar_wait_bounded(smem_u32(&full[j % kNS]), (j / kNS) & 1, &never, kTimeoutNs);
        if (nq > 0) mbar_wait_bounded(smem_u32(&bars->q_full), (nq - 1) & 1, &never, kTimeoutNs);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------- MMA issuers
      // warp 1 issues tile A's MMAs, warp 3 tile B's. S runs one used block
      // ahead of P.V, so S_X(j+1) overlaps the softmax of block j. The
      // counters gb (blocks), jS and jP (blocks this tile used) run on across
      // pairs, as do the barrier phases they select.
      const int x = warp == 1 ? 0 : 1;
      const bool leader = elect_one();
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idPV = idesc_bf16_f32(BM, D, true);
      const uint64_t dq = sdesc_sw128(sQ + x * kTile, 16, 1024);
      const uint64_t dk = sdesc_sw128(sK, 16, 1024);
      const uint64_t dv = sdesc_sw128(sV, kTile, 1024);
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait_bounded(smem_u32(bar), parity, abort, kTimeoutNs);
        return __all_sync(0xffffffffu, ok);
      };
      auto wait2 = [&](uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb) -> bool {
        const bool lo = lane < 16;
        const bool ok = mbar_wait_bounded(smem_u32(lo ? a : b), lo ? pa : pb, abort, kTimeoutNs);
        return __all_sync(0xffffffffu, ok);
      };
      int gb = 0, jS = 0, jP = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int o;
        if (!read_pair(bars, k, abort, &o, leader) || o < 0) break;
        PairGeom g;
        g.set(o, p);
        if (!wait(&bars->q_full, k & 1)) break;
        tc_fence_after();
        PairSched ss, sp;
        int bs = 0, jPp = 0;
        // the S cursor: block bs, used by this tile or only released by it
        auto advance_s = [&]() -> bool {
          ss.next(g.n_depth, g.nb);
          const bool use = g.uses(x, ss);
          const int gs = gb + bs, st = gs % kNS;
          const bool okw = (use && jS >= 1)
                               ? wait2(&bars->k_full[st], (gs / kNS) & 1, &bars->s_free[x], (jS - 1) & 1)
                               : wait(&bars->k_full[st], (gs / kNS) & 1);
          if (!okw) return false;
          tc_fence_after();
          if (use) {
            if (leader) {
              const uint64_t dks = dk + (uint64_t)((st * kTile) >> 4);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tbase + kColS + x * 128, dq + (uint64_t)(kk * 2), dks + (uint64_t)(kk * 2), idS,
                       kk > 0);
              tc_commit(smem_u32(&bars->k_empty[st]));
              tc_commit(smem_u32(&bars->s_full[x]));
            }
            ++jS;
          } else if (leader) {
            mbar_arrive(smem_u32(&bars->k_empty[st]));
          }
          __syncwarp();
          ++bs;
          return true;
        };
        // The S cursor stays at most two blocks ahead of the P.V cursor: S of
        // block bp+1 (when this tile uses it) goes out before P.V of block bp,
        // and no cursor ever waits for a block the rings cannot hold yet (a tile
        // whose next used block lies far ahead would otherwise hold back the
        // stages the other tile needs).
        for (int bp = 0; ok && bp < g.nb; ++bp) {
          while (ok && bs < g.nb && bs <= bp + 1) ok = advance_s();
          if (!ok) break;
          sp.next(g.n_depth, g.nb);
          const bool use = g.uses(x, sp);
          const int gv = gb + bp, st = gv % kNS;
          if (use) {
            if (!wait2(&bars->p_full[x], jP & 1, &bars->v_full[st], (gv / kNS) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (leader) {
              // the pair's first P.V of this tile overwrites O (the softmax
              // warps read the previous pair's O before they stored this P)
              const uint64_t dvs = dv + (uint64_t)((st * kTile) >> 4);
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_ts(tbase + kColO + x * 64, tbase + kColP + x * 64 + kk * 8,
                       dvs + (uint64_t)((kk * 2048) >> 4), idPV, (jPp > 0 || kk > 0) ? 1u : 0u);
              tc_commit(smem_u32(&bars->v_empty[st]));
              tc_commit(smem_u32(&bars->pv_done[x]));
            }
            __syncwarp();
            ++jP;
            ++jPp;
          } else {
            if (!wait(&bars->v_full[st], (gv / kNS) & 1)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive(smem_u32(&bars->v_empty[st]));
            __syncwarp();
          }
        }
        while (ok && bs < g.nb) ok = advance_s();  // release the remaining K stages
        if (!ok) break;
        // Q of this pair is free once every S product issued here has completed
        if (leader) tc_commit(smem_u32(&bars->q_free));
        __syncwarp();
        gb += g.nb;
      }
      if (leader) {
        int never = 0;
        tc_commit(smem_u32(&bars->mma_done[x]));
        mbar_wait_bounded(smem_u32(&bars->mma_done[x]), 0, &never, kTimeoutNs);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;\n" ::: "memory");
    // ---------------------------------------------------- softmax + epilogue
    const int tx = (warp - 4) >> 2;  // tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const int lp = row >> p.lgG;
    const int wq = warp & 3;  // this warp's word of a depth block
    const int lpw = (row & 31) >> p.lgG;
    const float sl = p.scale_log2;
    const uint32_t colS = kColS + tx * 128, colO = kColO + tx * 64, colP = kColP + tx * 64;
    const uint32_t zeros[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    bool p_zero = false;  // this warp's P columns outside its depth word hold zeros
    int j = 0;            // blocks of this tile so far, over all pairs
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int o;
      if (!read_pair(bars, k, abort, &o, lane == 0) || o < 0) break;
      PairGeom g;
      g.set(o, p);
      if (g.npos[tx] == 0) continue;  // tile B of a head's last pair may be absent
      const int p0x = g.p0 + tx * g.P;
      const int t_row = p0x + lp;
      const int h_row = g.hk * G + (row & (G - 1));
      const bool valid = lp < g.npos[tx];
      const int t_mask = min(t_row, p.T - 1);
      const int dw_lo = ((row & 31) >> p.lgG) * p.L;  // the row's slots among its warp's rows
      const int dw_n = valid ? p.L : 0;               // rows past T keep no depth column
      // layer-major words: column c holds position c % PW of the warp's
      // positions, slot index*(32/PW) + c / PW; this row's columns are
      // c = its position + i*PW
      const uint32_t lm_pat = g.PW >= 32 ? 1u << lpw : (0xffffffffu / ((1u << g.PW) - 1u)) << lpw;
      float m_ref = -INFINITY, l = 0.f;
      int jp = 0;  // blocks of this tile in this pair
      // Rescale O and l to a new reference when a block's raw max mx (log2
      // units) rose more than the threshold above it; false on a timeout.
      // O holds this pair's blocks 0..jp-1 of the tile (nothing when jp == 0).
      auto rescale = [&](float mx) -> bool {
        const bool need = mx > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mx : m_ref;
          const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
          if (jp > 0) {
            if (!warp_wait(smem_u32(&bars->pv_done[tx]), (j - 1) & 1, abort)) return false;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              const uint32_t ta = tmem_addr(tbase, lane_base, colO + c * 32);
              tmem_ld32(ta, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32(ta, r);
            }
            tmem_st_wait();
          }
          l *= alpha;
          m_ref = m_new;
        }
        return true;
      };
      // stale-reference fast path checked by the block sum (every p is at most
      // the sum, so a sum within 2^threshold proves the max did not rise past
      // it); max-first slow path with a lazy rescale of O and l (as in the
      // d = 128 kernel)
      PairSched sch;
      for (int b = 0; ok && b < g.nb; ++b) {
        sch.next(g.n_depth, g.nb);
        if (!g.uses(tx, sch)) continue;
        if (!warp_wait(smem_u32(&bars->s_full[tx]), j & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pcol = tmem_addr(tbase, lane_base, colP);
        float sum = 0.f;
        if (sch.depth) {
          // depth block: only this warp's word of 32 columns holds its rows'
          // slots; the row keeps its own [lo, hi) (a bit test and a select)
          uint32_t xs[32];
          tmem_ld32(tmem_addr(tbase, lane_base, colS + wq * 32), xs);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->s_free[tx]));
          uint32_t word;
          if (p.depth_lm) {
            const int SP = 32 / g.PW;
            const int nbits = min(SP, p.L - g.depth_index(sch.index) * SP) * g.PW;  // slots < L
            word = valid ? lm_pat & (nbits >= 32 ? 0xffffffffu : (1u << nbits) - 1u) : 0u;
          } else {
            const int lo = dw_lo - g.depth_index(sch.index) * 32, hi = lo + dw_n;
            const int a = min(max(lo, 0), 32), bb = min(max(hi, 0), 32);
            word = (bb >= 32 ? 0xffffffffu : (1u << bb) - 1u) & ~(a >= 32 ? 0xffffffffu : (1u << a) - 1u);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) xs[i] = (word & (1u << i)) ? xs[i] : 0xff800000u;  // -inf
          uint32_t pk[16];
          bool slow = __any_sync(0xffffffffu, m_ref == -INFINITY);
          if (!slow) {
            sum = exp_block<32>(xs, pk, sl, m_ref);
            slow = __any_sync(0xffffffffu, !(sum <= kSumBound));
          }
          if (slow) {
            if (!rescale(raw_max32(xs) * sl)) {
              ok = false;
              break;
            }
            sum = exp_block<32>(xs, pk, sl, m_ref);
          }
          l += sum;
          // the tile's P columns hold P of its previous block until that P.V is done
          if (j >= 1) {
            if (!warp_wait(smem_u32(&bars->pv_done[tx]), (j - 1) & 1, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          tmem_st16(pcol + wq * 16, pk);
          if (!p_zero) {
            for (int kk = 1; kk < 4; ++kk) tmem_st16(pcol + ((wq + kk) & 3) * 16, zeros);
          }
          p_zero = true;
        } else {
          uint32_t x[BN];
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) tmem_ld32(tmem_addr(tbase, lane_base, colS + c * 32), x + c * 32);
          tmem_ld_wait();
          // S is in registers: the tile's S columns may take its next block
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->s_free[tx]));
          // sequence block: the grouped causal mask keeps columns below hi
          const int k0 = sch.index * BN;
          if (k0 + BN - 1 > p0x) {
            const int hi = t_mask - k0 + 1;
#pragma unroll
            for (int c = 0; c < BN; ++c) x[c] = c < hi ? x[c] : 0xff800000u;  // -inf
          }
          uint32_t pk[BN / 2];
          bool slow = __any_sync(0xffffffffu, m_ref == -INFINITY);
          if (!slow) {
            sum = exp_block<BN>(x, pk, sl, m_ref);
            slow = __any_sync(0xffffffffu, !(sum <= kSumBound));
          }
          if (slow) {
            if (!rescale(raw_max128(x) * sl)) {
              ok = false;
              break;
            }
            sum = exp_block<BN>(x, pk, sl, m_ref);
          }
          l += sum;
          // the tile's P columns hold P of its previous block until that P.V is done
          if (j >= 1) {
            if (!warp_wait(smem_u32(&bars->pv_done[tx]), (j - 1) & 1, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tmem_st32(pcol + c * 32, pk + c * 32);
          p_zero = false;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->p_full[tx]));
        ++j;
        ++jp;
      }
      if (!ok) break;
      // epilogue: O holds every block of the tile once its last P.V is done
      // (commits complete in issue order). The next pair's first P.V of this
      // tile, which overwrites O, follows this warp's next p_full arrival.
      if (!warp_wait(smem_u32(&bars->pv_done[tx]), (j - 1) & 1, abort)) break;
      tc_fence_after();
      const float inv = 1.f / l;
      __nv_bfloat16* orow = p.o + ((int64_t)t_row * p.Hq + h_row) * D;
      uint32_t r[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem_addr(tbase, lane_base, colO + c * 32), r + c * 32);
      tmem_ld_wait();
      tc_fence_before();
      if (valid) {
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w[i] = pack_bf16x2(__uint_as_float(r[16 * c + 2 * i]) * inv, __uint_as_float(r[16 * c + 2 * i + 1]) * inv);
          if (p.o_v8) {
            st_global_v8(orow + 16 * c, w);
          } else {
            reinterpret_cast<uint4*>(orow)[2 * c] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4*>(orow)[2 * c + 1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
      if (valid && p.lse) p.lse[(int64_t)t_row * p.Hq + h_row] = m_ref * kLn2 + logf(l);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (tid == 0) {
    if (bars->abort) atomicCAS(p.err, 0u, (unsigned int)MODA_ERR_TIMEOUT);
    // the last CTA to finish puts the queue back to zero for the next launch
    __threadfence();
    if (atomicAdd(p.queue + 1, 1u) == gridDim.x - 1) {
      p.queue[0] = 0u;
      p.queue[1] = 0u;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_fwd_pp(const FwdArgs& a, cudaStream_t stream) {
  if (a.d != D) return cudaErrorInvalidValue;
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int P = BM >> lgG;
  const int ntiles = (a.T + P - 1) / P;
  const int npairs = (ntiles + 1) / 2;
  CUtensorMap tq, tk, tv, tkd, tvd;
  const uint64_t row = (uint64_t)D * 2;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)a.T};
    const uint64_t str[2] = {row, row * a.Hq};
    const uint32_t box[3] = {64, (uint32_t)a.G, (uint32_t)P};
    if (encode_bf16_sw128(&tq, a.q, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hk, (uint64_t)a.T};
    const uint64_t str[2] = {row, row * a.Hk};
    const uint32_t box[3] = {64, 1, BN};
    if (encode_bf16_sw128(&tk, a.k, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tv, a.v, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  if (a.L > 0 && a.layer_major) {
    // [L, T, Hk, d]: a box is one softmax warp's word, PW positions x 32/PW slots
    const uint32_t PW = (uint32_t)(P >> 2);
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)a.Hk, (uint64_t)a.T, (uint64_t)a.L};
    const uint64_t str[3] = {row, row * a.Hk, row * a.Hk * a.T};
    const uint32_t box[4] = {64, 1, PW, 32 / PW};
    // a depth row is 128 bytes here; the next 128 belong to another KV head,
    // read by other CTAs at other times: fetch 128-byte granules
    if (encode_bf16_sw128(&tkd, a.kd, 4, dims, str, box, 128) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tvd, a.vd, 4, dims, str, box, 128) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else if (a.L > 0) {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)a.Hk * a.T * a.L};
    const uint64_t str[1] = {row};
    const uint32_t box[2] = {64, 32};  // one softmax warp's word of a depth block
    if (encode_bf16_sw128(&tkd, a.kd, 2, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tvd, a.vd, 2, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else {
    tkd = tk;  // never read when L == 0
    tvd = tv;
  }
  PpParams prm;
  prm.T = a.T; prm.Hq = a.Hq; prm.Hk = a.Hk; prm.L = a.L; prm.lgG = lgG; prm.npairs = npairs;
  prm.depth_lm = a.layer_major;
  prm.scale_log2 = a.scale * kLog2e;
  prm.o = (__nv_bfloat16*)a.o;
  prm.o_v8 = ((uintptr_t)a.o & 31u) == 0;
  prm.lse = a.lse;
  prm.err = a.err;
  prm.total = npairs * a.Hk;
  prm.queue = a.queue;
  cudaError_t e = cudaFuncSetAttribute(moda_fwd_pp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  // one CTA per SM (each takes pairs from the queue until it is empty)
  const int grid = min(prm.total, a.num_sms > 0 ? a.num_sms : 148);
  moda_fwd_pp_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, tkd, tvd, prm);
  return cudaGetLastError();
}

}  // namespace moda
