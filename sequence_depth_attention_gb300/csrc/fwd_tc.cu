// MoDA forward on the 5th-generation tensor core (sm_103a): TMA-staged tiles,
// tcgen05.mma into tensor memory (TMEM), warp-specialised pipeline, one
// persistent CTA per SM. This kernel serves d = 128; d = 64 runs two tiles per
// CTA (fwd_pp.cu).
//
// What it computes is Mixture-of-Depths Attention, Sec. 2.2 (one softmax over
// the causal sequence keys of the layer and the L depth slots of the same
// position), organised as the paper's fused kernel (Sec. 3.3, Algorithm 1):
//
//   * group-aware query tile (Sec. 3.2): the M = 128 rows of a tile are 128/G
//     consecutive positions x the G query heads that share KV head hk, row
//     r <-> (position p0 + r/G, head hk*G + r%G). One 3-D TMA box over
//     q[T][Hq][d] lands exactly this stacking, so every K/V block staged in
//     shared memory serves all G heads;
//   * depth blocks: the packed depth rows of the tile's positions are one
//     contiguous run kd[hk][p0 .. p0+128/G)[0..L) (chunk-aware layout). Each
//     softmax warp owns one 32-row word of every depth block, filled with the
//     next packed rows of its own positions, so a row keeps depth columns of
//     its own warp's word only (the block-diagonal mask of Sec. 3.3 within
//     that word). From layer-major depth tensors [L][T][Hk][d] (the order the
//     layers write them) the copy engine gathers the same word shape itself:
//     a 4-D box of the warp's PW positions x 32/PW slots, so the chunk-aware
//     grouping needs no relayout pass; a row's columns are then every PW-th
//     one. An exact online softmax does not depend on block order, so depth
//     blocks are spread evenly among the sequence blocks: each tile streams
//     its depth rows from HBM over its lifetime;
//   * sequence blocks of 128 keys, the grouped causal mask key <= p0 + r/G
//     applied only on blocks that reach past p0;
//   * one running state per row: max m (log2 units), sum l, and the
//     unnormalised output O, which lives in TMEM and is accumulated by the
//     tensor core; o = O / l once at the end, lse = m ln2 + ln l.
//
// Persistent CTAs: the grid is one CTA per SM, and each CTA takes tiles from
// a queue in global memory, longest tiles first (KV-head-major once the K/V
// of all heads overflow half of L2). The pipeline runs on
// across tile boundaries: the next tile's Q and K/V blocks load while the
// current one finishes, its first S = Q K^T products run during the current
// tile's last block and epilogue, so a tile costs no launch, prologue or
// pipeline drain. The K-producer warp takes tiles from the queue and passes
// their numbers to the other roles through a ring in shared memory.
//
// Roles (8 warps):
//   warp 0  lane 0: tile queue, TMA producer for Q and the K blocks
//   warp 1  lane 0: tcgen05.mma issuer of S = Q K^T; the whole warp allocates TMEM
//   warp 2  lane 0: TMA producer for the V blocks
//   warp 3  lane 0: tcgen05.mma issuer of O += P V
//   warps 4-7     : softmax, one thread per tile row (= TMEM lane), the copy
//                   of each tile's Q into TMEM, and the epilogue
// TMEM (512 columns): S double buffer [0,128) [128,256), O [256, 256+d),
// P (bf16 pairs) [384,448), Q (bf16 pairs) [448, 448+d/2). The softmax warps
// copy each tile's Q rows from shared memory into TMEM once the previous
// tile's last S = Q K^T has completed, so S reads only K from shared memory
// (an MMA with both operands in shared memory would use the whole
// shared-memory read bandwidth and starve the TMA writes of the next K/V
// blocks). The MMA computes S_{j+1} = Q K_{j+1}^T while the softmax turns S_j
// into P_j, then O += P_j V_j with P read straight from TMEM.
// The running max is rescaled lazily: O and l are rescaled only when a new
// block raises the row max by more than 8 (a factor 256), which stays exact
// because o = O / l uses the same reference for both.
//
// Every wait is bounded (2 s); on expiry the CTA stops issuing work, waits
// for its in-flight copies and MMAs, frees TMEM and latches MODA_ERR_TIMEOUT
// in the device error word.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "softmax_block.cuh"
#include "tensor_map.h"

namespace moda {
namespace {

using namespace sm103;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 256;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kSumBound = 256.0f;         // 2^kRescaleThreshold
constexpr int kTileRing = 4;                // tile numbers in flight between roles
// arrivals that free a tile-ring entry: V producer, S issuer, P.V issuer, 4 softmax warps
constexpr int kTileReaders = 7;

template <int D>
struct Cfg {
  static constexpr int kBoxes = D / 64;     // 64-column (128-byte) swizzle boxes per row
  static constexpr int kBoxBytes = 128 * 64 * 2;
  static_assert(D == 128, "d = 64 runs the two-tile kernel (fwd_pp.cu)");
  static constexpr int kNSK = 3;  // K stages
  static constexpr int kNSV = 3;  // V stages
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kNSK * kKVBytes;
  static constexpr int kOffBar = kOffV + kNSV * kKVBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384, kColQ = 448;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct alignas(8) Barriers {
  uint64_t q_full, q_tmem;  // Q of the current tile landed / copied into TMEM
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t t_full[kTileRing], t_empty[kTileRing];
  uint64_t mma_done, mma_done_pv;
  uint64_t o_staged;  // a tile's O rows sit in the Q region (128 softmax arrivals)
  uint64_t o_free;    // the TMA store of that O has read the Q region
  int tile_ring[kTileRing];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Barriers) <= 512, "barrier block");

struct Params {
  int T, Hq, Hk, L, lgG, ntiles, total, head_major;
  int depth_lm;  // depth K/V layer-major [L, T, Hk, d] (else packed [Hk, T, L, d])
  float scale_log2;
  float* lse;
  unsigned int* err;
  unsigned int* queue;  // {next tile, CTAs finished}
};

// All lanes poll; the warp proceeds only if every lane saw the phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

// Geometry of one tile. Queue entry o: longest tiles first; KV-head-major
// when the heads' K/V together overflow half of L2 (resident tiles then share
// one or two heads' K/V), else heads interleaved (longest first over all
// heads, which balances the last wave better when every head's K/V stays in
// L2 anyway).
struct Tile {
  int hk, p0, npos, t_last, PW, RW, n_depth, nb, depth_row0;
  __device__ void set(int o, const Params& p) {
    const int P = BM >> p.lgG;  // positions per tile
    const int tile = p.ntiles - 1 - (p.head_major ? o % p.ntiles : o / p.Hk);
    hk = p.head_major ? o / p.ntiles : o % p.Hk;
    p0 = tile * P;
    npos = min(P, p.T - p0);
    t_last = p0 + npos - 1;
    PW = P >> 2;                     // positions per softmax warp
    RW = PW * p.L;                   // packed depth rows per softmax warp
    // a word holds 32 rows: 32 consecutive packed rows, or (layer-major) PW
    // positions x 32/PW slots
    n_depth = ((p.depth_lm ? PW : min(npos, PW)) * p.L + 31) / 32;
    nb = n_depth + t_last / BN + 1;
    depth_row0 = (hk * p.T + p0) * p.L;
  }
};

// Block schedule of a tile: the n_depth depth blocks are spread evenly among
// the sequence blocks (Bresenham: block j is a depth block iff
// floor((j+1)*n_depth/nb) > floor(j*n_depth/nb)). Every role walks the blocks
// in order with its own copy.
struct Sched {
  int acc = 0, db = 0, sbk = 0;  // remainder, depth blocks so far, sequence blocks so far
  bool depth = false;            // is the current block a depth block
  int index = 0;                 // its index among blocks of its kind
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

// The k-th tile of this CTA from the ring (-1: no more tiles); the reader
// frees the entry right away. False on a timeout.
__device__ __forceinline__ bool read_tile(Barriers* bars, int k, volatile int* abort, int* o,
                                          bool arrive) {
  const int s = k % kTileRing;
  if (!warp_wait(smem_u32(&bars->t_full[s]), (k / kTileRing) & 1, abort)) return false;
  *o = *reinterpret_cast<volatile int*>(&bars->tile_ring[s]);
  __syncwarp();
  if (arrive) mbar_arrive(smem_u32(&bars->t_empty[s]));
  return true;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
moda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKd,
                   const __grid_constant__ CUtensorMap tmVd, const __grid_constant__ CUtensorMap tmO,
                   const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kOffBar);
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  volatile int* abort = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = 1 << p.lgG;

  if (tid == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_tmem), 128);
    mbar_init(smem_u32(&bars->o_staged), 128);
    mbar_init(smem_u32(&bars->o_free), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->k_empty[s]), 1);
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->s_full[b]), 1);
      mbar_init(smem_u32(&bars->s_free[b]), 128);
      mbar_init(smem_u32(&bars->p_full[b]), 128);
      mbar_init(smem_u32(&bars->pv_done[b]), 1);
    }
    for (int s = 0; s < kTileRing; ++s) {
      mbar_init(smem_u32(&bars->t_full[s]), 1);
      mbar_init(smem_u32(&bars->t_empty[s]), kTileReaders);
    }
    mbar_init(smem_u32(&bars->mma_done), 1);
    mbar_init(smem_u32(&bars->mma_done_pv), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
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

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------ TMA producers
    // The whole warp runs the loop (uniform control flow); one elected lane
    // issues the copies. Stages and phases follow the CTA's running block
    // count g across tiles.
    const bool leader = elect_one();
    const bool is_k = warp == 0;
    const int NS = is_k ? C::kNSK : C::kNSV;
    const uint32_t sbase = is_k ? sK : sV;
    const CUtensorMap* seq_map = is_k ? &tmK : &tmV;
    const CUtensorMap* dep_map = is_k ? &tmKd : &tmVd;
    uint64_t* full = is_k ? bars->k_full : bars->v_full;
    uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
    // Q and the depth rows are read once: evict them first so they do not
    // push the K/V blocks that later tiles of the head re-read out of L2
    // (K/V keep the default policy; pinning all of them measured slower).
    const uint64_t pol_once = l2_policy_evict_first();
    int g = 0;   // blocks issued so far, over all tiles
    int nq = 0;  // Q loads issued
    int ntile = 0;            // tiles taken (K producer)
    int tile_even = 0, tile_odd = 0;  // the last two tiles' numbers (K producer)
    // The O of tile kk: the softmax warps stage its rows in the Q region (in
    // the o tensor map's box layout) once the next tile's Q is in TMEM; one
    // TMA store per 64-column half writes them out, and the region is free
    // again once the store has read it.
    auto store_o = [&](int kk) -> bool {
      if (!warp_wait(smem_u32(&bars->o_staged), kk & 1, abort)) return false;
      if (leader) {
        Tile t;
        t.set((kk & 1) ? tile_odd : tile_even, p);
        for (int c = 0; c < C::kBoxes; ++c) tma_store_3d(&tmO, sQ + c * C::kBoxBytes, c * 64, t.hk * G, t.p0);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(smem_u32(&bars->o_free));
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int o;
      if (is_k) {
        // take the next tile from the queue and pass it on
        const int s = k % kTileRing;
        if (!warp_wait(smem_u32(&bars->t_empty[s]), ((k / kTileRing) & 1) ^ 1, abort)) break;
        if (leader) {
          const unsigned int t = atomicAdd(p.queue, 1u);
          o = t < (unsigned int)p.total ? (int)t : -1;
          *reinterpret_cast<volatile int*>(&bars->tile_ring[s]) = o;
          mbar_arrive(smem_u32(&bars->t_full[s]));
        }
        o = __shfl_sync(0xffffffffu, o, __ffs(__ballot_sync(0xffffffffu, leader)) - 1);
      } else if (!read_tile(bars, k, abort, &o, leader)) {
        break;
      }
      if (o < 0) break;
      Tile tl;
      tl.set(o, p);
      if (is_k) {
        // Q of this tile, once the softmax warps have copied the previous Q
        // into TMEM and the O of tile k-2, staged in the Q region after that
        // copy, has been read out of it
        if (k > 0 && !warp_wait(smem_u32(&bars->q_tmem), (k - 1) & 1, abort)) break;
        if (k >= 2 && !store_o(k - 2)) break;
        if (k & 1) tile_odd = o; else tile_even = o;
        ntile = k + 1;
        if (leader) {
          const uint32_t qb = smem_u32(&bars->q_full);
          mbar_arrive_expect_tx(qb, C::kQBytes);
          for (int c = 0; c < C::kBoxes; ++c)
            tma_load_3d_hint(sQ + c * C::kBoxBytes, &tmQ, qb, c * 64, tl.hk * G, tl.p0, pol_once);
        }
        ++nq;
      }
      Sched sch;
      for (int j = 0; j < tl.nb; ++j, ++g) {
        sch.next(tl.n_depth, tl.nb);
        const int s = g % NS;
        if (!warp_wait(smem_u32(&empty[s]), ((g / NS) & 1) ^ 1, abort)) {
          ok = false;
          break;
        }
        if (leader) {
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, C::kKVBytes);
          const uint32_t dst = sbase + s * C::kKVBytes;
          if (sch.depth) {
            // four 32-row words: rows [32w, 32w+32) of the stage hold warp w's
            // packed depth rows 32*index .. +32 (128-byte swizzle atoms are 8
            // rows, so a word starts on an atom boundary). Layer-major depth:
            // the copy gathers the same word shape itself, slots
            // [SP*index, SP*index + SP) of warp w's PW positions, row
            // l_local*PW + t_local (SP = 32/PW)
            if (p.depth_lm) {
              const int SP = 32 / tl.PW;
              for (int w = 0; w < 4; ++w)
                for (int c = 0; c < C::kBoxes; ++c)
                  tma_load_4d_hint(dst + c * C::kBoxBytes + w * 32 * 128, dep_map, fb, c * 64, tl.hk,
                                   tl.p0 + w * tl.PW, sch.index * SP, pol_once);
            } else {
              for (int w = 0; w < 4; ++w)
                for (int c = 0; c < C::kBoxes; ++c)
                  tma_load_2d_hint(dst + c * C::kBoxBytes + w * 32 * 128, dep_map, fb, c * 64,
                                   tl.depth_row0 + w * tl.RW + sch.index * 32, pol_once);
            }
          } else {
            for (int c = 0; c < C::kBoxes; ++c)
              tma_load_3d(dst + c * C::kBoxBytes, seq_map, fb, c * 64, tl.hk, sch.index * BN);
          }
        }
        __syncwarp();
      }
    }
    // the last two tiles' O (nothing to wait for after a timeout: the
    // bounded waits return at once once the abort flag is up)
    if (is_k)
      for (int kk = max(0, ntile - 2); kk < ntile && !*abort; ++kk)
        if (!store_o(kk)) break;
    // drain: every copy this warp issued has landed (and every O store has
    // completed) before smem is released
    if (leader) {
      if (is_k) bulk_wait_group0();
      int never = 0;
      for (int j = max(0, g - NS); j < g; ++j)
        mbar_wait_bounded(smem_u32(&full[j % NS]), (j / NS) & 1, &never, kTimeoutNs);
      if (is_k && nq > 0) mbar_wait_bounded(smem_u32(&bars->q_full), (nq - 1) & 1, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------ MMA issuers
    // Warp 1 issues the S = Q K^T products, warp 3 the O += P V products.
    // Each waits for its own operands and commits its own MMAs, so the
    // waits and fences of one overlap the other's MMAs on the tensor core.
    // One elected thread of each runs its whole schedule, waits included:
    // the tensor core queues few MMAs, so every instruction between two
    // MMAs can leave it idle, and the softmax warps share the issue slots.
    if (elect_one()) {
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return mbar_wait_bounded(smem_u32(bar), parity, abort, kTimeoutNs);
      };
      auto next_tile = [&](int k, int* o) -> bool {
        const int s = k % kTileRing;
        if (!wait(&bars->t_full[s], (k / kTileRing) & 1)) return false;
        *o = *reinterpret_cast<volatile int*>(&bars->tile_ring[s]);
        mbar_arrive(smem_u32(&bars->t_empty[s]));
        return true;
      };
      // all descriptors here share the high word (SBO 1024, 128-byte swizzle);
      // tile offsets are 32-bit adds to the start address field of the low word
      const uint64_t dk = sdesc_sw128(sK, 16, 1024);
      const uint32_t hi = (uint32_t)(dk >> 32);
      int g = 0;  // blocks issued so far, over all tiles
      if (warp == 1) {
        constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false);
        const uint32_t k_lo = (uint32_t)dk;
        // S_g = Q K_g^T into S buffer g&1 as soon as the softmax has read
        // S_{g-2} out of that buffer and K_g has landed: S_{g+2} runs on the
        // tensor core while the softmax works on g. A tile's first S also
        // waits until the tile's Q sits in TMEM.
        bool ok = true;
        for (int k = 0; ok; ++k) {
          int o;
          if (!next_tile(k, &o) || o < 0) break;
          Tile tl;
          tl.set(o, p);
          if (!wait(&bars->q_tmem, k & 1)) break;
          for (int j = 0; j < tl.nb; ++j, ++g) {
            const int ks = g % C::kNSK;
            if (g >= 2 && !wait(&bars->s_free[g & 1], ((g - 2) >> 1) & 1)) {
              ok = false;
              break;
            }
            if (!wait(&bars->k_full[ks], (g / C::kNSK) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t kb = k_lo + ((uint32_t)(ks * C::kKVBytes) >> 4);
            const uint32_t dcol = tbase + C::kColS + (g & 1) * 128;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
              mma_ts(dcol, tbase + C::kColQ + kk * 8, desc_join(kb + off, hi), idS, kk > 0);
            }
            tc_commit(smem_u32(&bars->k_empty[ks]));
            tc_commit(smem_u32(&bars->s_full[g & 1]));
          }
        }
      } else {
        constexpr uint32_t idPV = idesc_bf16_f32(BM, D, true);
        const uint32_t v_lo = (uint32_t)sdesc_sw128(sV, C::kBoxBytes, 1024);
        const uint32_t pcol = tbase + C::kColP;
        bool ok = true;
        for (int k = 0; ok; ++k) {
          int o;
          if (!next_tile(k, &o) || o < 0) break;
          Tile tl;
          tl.set(o, p);
          for (int j = 0; j < tl.nb; ++j, ++g) {
            const int sb = g & 1, vs = g % C::kNSV;
            if (!wait(&bars->p_full[sb], (g >> 1) & 1) || !wait(&bars->v_full[vs], (g / C::kNSV) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t vb = v_lo + ((uint32_t)(vs * C::kKVBytes) >> 4);
            // a tile's first P.V overwrites O (the softmax warps have read the
            // previous tile's O before they stored this P)
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts(tbase + C::kColO, pcol + kk * 8, desc_join(vb + ((uint32_t)(kk * 2048) >> 4), hi),
                     idPV, kk > 0 ? 1u : acc0);
            tc_commit(smem_u32(&bars->v_empty[vs]));
            tc_commit(smem_u32(&bars->pv_done[sb]));
          }
        }
      }
      // every MMA issued by this thread has completed before TMEM is freed
      uint64_t* done = warp == 1 ? &bars->mma_done : &bars->mma_done_pv;
      int never = 0;
      tc_commit(smem_u32(done));
      mbar_wait_bounded(smem_u32(done), 0, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------ softmax + epilogue
    const int row = tid - 128;                 // tile row == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const int wq = warp & 3;                    // this warp's word of a depth block
    const int lp = row >> p.lgG;
    const int h_off = row & (G - 1);
    const float sl = p.scale_log2;
    const uint32_t zeros[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    bool p_zero = false;  // this warp's P columns outside its depth word hold zeros
    int g = 0;            // blocks processed so far, over all tiles
    bool ok = true;
    // Q of tile k (landed in shared memory) -> TMEM columns [kColQ, kColQ + d/2)
    // as bf16 pairs in row order, the A operand of S = Q K^T. Called once
    // every S product of the previous tile has completed.
    auto copy_q = [&](int k) -> bool {
      if (!warp_wait(smem_u32(&bars->q_full), k & 1, abort)) return false;
      const uint8_t* qrow = smem + C::kOffQ + row * 128;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(qrow + c * C::kBoxBytes + ((i ^ (row & 7)) << 4));
          w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
        tmem_st32(tmem_addr(tbase, lane_base, C::kColQ + c * 32), w);
      }
      tmem_st_wait();
      tc_fence_before();
      // the Q region takes the next tile's Q (a TMA write): order these reads first
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(smem_u32(&bars->q_tmem));
      return true;
    };
    int o_cur;
    ok = read_tile(bars, 0, abort, &o_cur, lane == 0);
    if (ok && o_cur >= 0) ok = copy_q(0);
    for (int k = 0; ok && o_cur >= 0; ++k) {
      Tile tl;
      tl.set(o_cur, p);
      // After the tile's last block (its S has been read, so every S product
      // that used this tile's Q has completed), the next tile's number is
      // read from the ring (the K producer publishes it after this tile's
      // last K load) and its Q goes into TMEM, so that its first S products
      // run while this tile's last P.V completes and its epilogue runs.
      int o_next = -1;
      auto prepare_next = [&]() -> bool {
        if (!read_tile(bars, k + 1, abort, &o_next, lane == 0)) return false;
        return o_next < 0 || copy_q(k + 1);
      };
      const int t_row = tl.p0 + lp;
      const int h_row = tl.hk * G + h_off;
      const bool valid = t_row < p.T;
      const int t_mask = min(t_row, p.T - 1);
      const int dw_lo = ((row & 31) >> p.lgG) * p.L;  // the row's slots among its warp's RW rows
      const int dw_n = valid ? p.L : 0;             // rows past T keep no depth column
      // layer-major words: column c holds position c % PW of the warp's
      // positions, slot index*(32/PW) + c / PW; this row's columns are
      // c = its position + i*PW
      const int lpw = (row & 31) >> p.lgG;
      const uint32_t lm_pat = tl.PW >= 32 ? 1u << lpw : (0xffffffffu / ((1u << tl.PW) - 1u)) << lpw;
      float m_ref = -INFINITY, l = 0.f;
      // Rescale O and l to a new reference when a block's raw max mx (log2
      // units) rose more than the threshold above it; false on a timeout.
      // O holds this tile's blocks 0..j-1 (nothing of it when j == 0).
      auto rescale = [&](float mx, int j) -> bool {
        const bool need = mx > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mx : m_ref;
          const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
          if (j > 0) {
            if (!warp_wait(smem_u32(&bars->pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort)) return false;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              const uint32_t ta = tmem_addr(tbase, lane_base, C::kColO + c * 32);
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
      // Fast path of every block: exponentiate against the running reference
      // m_ref right away. Every p is at most the block's sum, so a sum within
      // 2^threshold proves no score rose more than the threshold above m_ref,
      // and the block needs no max at all. Only if some row of the warp has no
      // reference yet, or its sum exceeds the bound, fall back to max-first
      // with a rescale of O and l where the max really rose that far.
      Sched sch;
      for (int j = 0; j < tl.nb; ++j, ++g) {
        sch.next(tl.n_depth, tl.nb);
        const int sb = g & 1;
        if (!warp_wait(smem_u32(&bars->s_full[sb]), (g >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pcol = tmem_addr(tbase, lane_base, C::kColP);
        float sum = 0.f;
        if (sch.depth) {
          // depth block: only this warp's word of 32 columns can hold its rows'
          // slots; mask (on raw scores, scale > 0) to the row's own slots with
          // one validity word, a bit test and a select per column
          uint32_t xs[32];
          tmem_ld32(tmem_addr(tbase, lane_base, C::kColS + sb * 128 + wq * 32), xs);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->s_free[sb]));
          uint32_t word;
          if (p.depth_lm) {
            const int SP = 32 / tl.PW;
            const int nbits = min(SP, p.L - sch.index * SP) * tl.PW;  // columns of slots < L
            word = valid ? lm_pat & (nbits >= 32 ? 0xffffffffu : (1u << nbits) - 1u) : 0u;
          } else {
            const int lo = dw_lo - sch.index * 32, hi = lo + dw_n;
            const int a = min(max(lo, 0), 32), b = min(max(hi, 0), 32);
            word = (b >= 32 ? 0xffffffffu : (1u << b) - 1u) & ~(a >= 32 ? 0xffffffffu : (1u << a) - 1u);
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
            if (!rescale(raw_max32(xs) * sl, j)) {
              ok = false;
              break;
            }
            sum = exp_block<32>(xs, pk, sl, m_ref);
          }
          l += sum;
          // P_g overwrites P_{g-1}: the tensor core must have consumed it
          if (g >= 1) {
            if (!warp_wait(smem_u32(&bars->pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort)) {
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
          // sequence block: S row of this thread, 128 raw fp32 scores as bits
          uint32_t x[BN];
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            tmem_ld32(tmem_addr(tbase, lane_base, C::kColS + sb * 128 + c * 32), x + c * 32);
          tmem_ld_wait();
          // S_g is in registers: its TMEM buffer may take S_{g+2}
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->s_free[sb]));
          // the grouped causal mask keeps columns below hi (on raw scores:
          // scale > 0, so masking and the max commute with scaling)
          const int k0 = sch.index * BN;
          if (k0 + BN - 1 > tl.p0) {
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
            if (!rescale(raw_max128(x) * sl, j)) {
              ok = false;
              break;
            }
            sum = exp_block<BN>(x, pk, sl, m_ref);
          }
          l += sum;
          // P_g overwrites P_{g-1}: the tensor core must have consumed it (the
          // slow path above may have waited for it already; the phase test is
          // idempotent)
          if (g >= 1) {
            if (!warp_wait(smem_u32(&bars->pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort)) {
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
        mbar_arrive(smem_u32(&bars->p_full[sb]));
      }
      if (!ok || !prepare_next()) break;
      // epilogue: O holds every block of the tile once the last P.V is done
      // (commits complete in issue order)
      if (!warp_wait(smem_u32(&bars->pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem_addr(tbase, lane_base, C::kColO + c * 32), r + c * 32);
      tmem_ld_wait();
      const float inv = 1.f / l;
      // The row of o goes into the Q region (the next tile's Q is in TMEM by
      // now) in the 128-byte-swizzled layout of the o tensor map's box, row
      // `row` of each 64-column half; the K-producer thread writes the tile
      // out with TMA stores, which skip the rows past T. The previous tile's
      // store must have read the region first (it has whenever a next tile's
      // Q was loaded into it; after the last tile it may still be reading).
      if (k > 0 && !warp_wait(smem_u32(&bars->o_free), (k - 1) & 1, abort)) {
        ok = false;
        break;
      }
      uint8_t* srow = smem + C::kOffQ + row * 128;
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            v[e] = pack_bf16x2(__uint_as_float(r[64 * c + 8 * i + 2 * e]) * inv,
                               __uint_as_float(r[64 * c + 8 * i + 2 * e + 1]) * inv);
          *reinterpret_cast<uint4*>(srow + c * C::kBoxBytes + ((i ^ (row & 7)) << 4)) =
              make_uint4(v[0], v[1], v[2], v[3]);
        }
      // the TMA store reads these bytes through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(smem_u32(&bars->o_staged));
      if (valid && p.lse) p.lse[(int64_t)t_row * p.Hq + h_row] = m_ref * kLn2 + logf(l);
      // O has been read: the next tile's first P.V may overwrite it (that
      // P.V follows this warp's next p_full arrival, so program order suffices)
      tc_fence_before();
      o_cur = o_next;
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

template <int D>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t stream) {
  using C = Cfg<D>;
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int P = BM >> lgG;
  const int ntiles = (a.T + P - 1) / P;
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
    if (encode_bf16_sw128(&tkd, a.kd, 4, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tvd, a.vd, 4, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
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
  CUtensorMap to;  // o [T][Hq][d]: the same boxes as q (a tile's rows, 64 columns each)
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)a.T};
    const uint64_t str[2] = {row, row * a.Hq};
    const uint32_t box[3] = {64, (uint32_t)a.G, (uint32_t)P};
    if (encode_bf16_sw128(&to, a.o, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  Params prm;
  prm.T = a.T; prm.Hq = a.Hq; prm.Hk = a.Hk; prm.L = a.L; prm.lgG = lgG; prm.ntiles = ntiles;
  prm.depth_lm = a.layer_major;
  prm.total = ntiles * a.Hk;
  // K and V of every KV head, bf16: head-major order once they overflow half of L2
  prm.head_major = (uint64_t)a.Hk * a.T * D * 2 * 2 > (64ull << 20) ? 1 : 0;
  prm.scale_log2 = a.scale * kLog2e;
  prm.lse = a.lse;
  prm.err = a.err;
  prm.queue = a.queue;
  cudaError_t e = cudaFuncSetAttribute(moda_fwd_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // one CTA per SM (each takes tiles from the queue until it is empty)
  const int grid = min(prm.total, a.num_sms > 0 ? a.num_sms : 148);
  moda_fwd_tc_kernel<D><<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tkd, tvd, to,
                                                                               prm);
  return cudaGetLastError();
}

}  // namespace

// d = 128 runs this kernel; d = 64 the two-tiles-per-CTA kernel of fwd_pp.cu.
cudaError_t launch_fwd_tc(const FwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_fwd_pp(a, stream);
}

}  // namespace moda
