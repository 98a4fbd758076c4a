// Backward pass of exact attention on sm_103a.
//
// The pages keep only O and the per-row statistics from the forward pass and
// compute the score and probability tiles again from Q, K and V ("FlashAttention and GPU
// Memory", chapter 09). With lse_i the row logsumexp, for a block of keys j
// and a block of queries i:
//   S = Q_i K_j^T,  P = exp(scale S - lse_i),  dP = dO_i V_j^T,
//   dS = P o (dP - D_i)   with D_i = dO_i . O_i,
//   dV_j += P^T dO_i,  dK_j += scale dS^T Q_i,  dQ_i += scale dS K_j.
// (The chain rule of softmax; D_i = sum_k P_ik dP_ik equals dO_i . O_i.)
//
// Three kernels run in order on one stream:
//   1. bwd_prep: D_i = dO_i . O_i in fp32 (the only workspace).
//   2. bwd_dkdv: one CTA per 128-key block, looping over 128-row query blocks;
//      accumulates dK and dV in tensor memory (TMEM).
//   3. bwd_dq:   one CTA per 128-row query block, looping over 128-key blocks;
//      accumulates dQ in TMEM.
// At d = 64 the dQ kernel runs first and forms D itself, from the dO tile it
// loads anyway and an O tile loaded beside it, and writes it for the dK/dV
// kernel after it: a small start kernel only resets the work counters, and dO
// is read from device memory twice instead of three times.
// Both main kernels rebuild S and dP; dQ is summed on chip in a fixed order,
// so the result is deterministic and no fp32 atomics are needed (on GB300 the
// L2's atomic-add rate, about 1.1-1.4e12 fp32 adds/s, would otherwise bound
// the pass).
//
// Warp roles in both main kernels: warpgroups 0 and 1 (warps 0-7) do the
// elementwise work, each on half of the block's columns (thread r owns TMEM
// lane r); warp 8 issues TMA loads; warp 9 issues the tcgen05 MMAs and owns the
// 512-column TMEM allocation; warp 10 issues the products that share no TMEM
// columns with warp 9's (S^T in the dK/dV kernel, dQ in the dQ kernel), so
// both kernels run 352 threads. P^T and dS^T (dK/dV kernel) and dS
// (dQ kernel) are written back into TMEM as bf16 over fp32 columns the
// warpgroups have already read, and used from there as the A operand of the
// next product. Each S or dP tile is released to the MMA warp as soon as the
// warpgroups hold it in registers, so the next tile's product overlaps their
// elementwise work.
//
// Template flags add per-sequence lengths (padding masks: each tile reads its
// sequence's lengths) and dropout (the forward's Philox mask made again from
// the seed, applied to P^T for dV and to dP in dS) without changing the plain
// kernels.
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_internal.h"
#include "block_order.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace fa::ptx;

constexpr float kLog2e = 1.44269504088896340736f;
constexpr int kPanelBytes = 128 * 128;  // 128 rows x 128 bytes (64 bf16)

// One 128-byte-swizzled row of a panel: 'nchunks' 16-byte chunks from chunk0.
__device__ __forceinline__ void st_swizzled_row(uint8_t* panel, int r, int chunk0, const uint32_t* w, int nchunks) {
#pragma unroll
  for (int c = 0; c < nchunks; ++c) {
    const int chunk = chunk0 + c;
    st_shared_v4(smem_u32(panel + r * 128 + (((chunk & 7) ^ (r & 7)) << 4)), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                 w[4 * c + 3]);
  }
}

// Reads 'ncols' fp32 TMEM columns of this thread's lane, scales, converts to
// bf16 and writes them to row r of a swizzled staging tile starting at
// feature column c0 (a multiple of 32).
template <int NCOLS>
__device__ __forceinline__ void stage_row_bf16(uint32_t taddr, uint8_t* tile, int r, int c0, float mul) {
#pragma unroll 1
  for (int c = 0; c < NCOLS; c += 32) {
    uint32_t o[32];
    tmem_ld32(taddr + c, o);
    tmem_ld_wait(o);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
    const int f = c0 + c;
    st_swizzled_row(tile + (f >> 6) * kPanelBytes, r, (f & 63) >> 3, w, 4);
  }
}

// ============================================================================ dK / dV
// Persistent: each CTA takes (head, 128-key block) tiles from a work counter
// until none is left. Within a tile, TMEM lane = key and each iteration covers
// 128 queries; warpgroup w handles queries [64 w, 64 w + 64) of each block and
// writes P^T and dS^T (bf16) over its own dP^T columns once it has read them.
//
// Across tiles the pipeline does not drain: the Q and dO rings and the S/dP/dS
// barriers count query blocks over the CTA's whole run, the next tile's K and
// V are loaded once this tile's last S^T and dP^T have read the buffers, and
// its first products run while the warpgroups write out this tile's dK and dV.
// The epilogue stages dV and dK as bf16 in the ring slots of the tile's last
// block; the producer warp stores them with TMA and then releases the slots.
template <int D>
struct DkdvCfg {
  static constexpr int BK = 128;  // keys per tile
  static constexpr int BQ = 128;  // queries per iteration
  static constexpr int kTileBytes = (D / 64) * kPanelBytes;
  // Q is needed first in each block (by S^T, two blocks ahead) and dO later
  // (by dP^T, one block ahead), so Q gets the deeper ring. Both slots of block
  // i are released together once its dV completes.
  static constexpr int kQStages = D == 128 ? 3 : 4;
  static constexpr int kDOStages = D == 128 ? 2 : 4;
  static_assert(kDOStages <= kQStages && kQStages <= 4, "the slot-release ring is indexed by Q slot");
  static constexpr int kItemSlots = 4;  // tiles fetched ahead by the producer
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffRow = kOffDO + kDOStages * kTileBytes;  // [parity][warpgroup][-lse(64) | -D(64)] fp32
  static constexpr int kOffBar = kOffRow + 2 * 2 * 128 * 4;
  // No alignment slack: the kernel checks that dynamic shared memory starts on
  // a 1024-byte boundary (the 128-byte swizzle atoms need it).
  static constexpr int kSmemBytes = kOffBar + 512;
  static constexpr uint32_t kColS = 0;     // S^T fp32
  static constexpr uint32_t kColDP = 128;  // dP^T fp32, then P^T and dS^T as bf16 over it (dkdv_pcol)
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
};

struct DkdvBarriers {
  uint64_t item_full[4], item_empty[4];     // tile ring: producer -> MMA warp and warpgroups
  uint64_t k_full, k_empty, v_full, v_empty;  // K and V buffers (one tile each)
  uint64_t q_full[4], do_full[4];
  // block b's Q and dO slots are free again: barrier b % kQStages, phase b / kQStages
  // (one commit after its dV; the producer arrives instead for a tile's last block)
  uint64_t blk_free[4];
  uint64_t s_full, s_free, dp_full, ds_half[2];
  uint64_t kv_done, teardown, teardown_s;  // a tile's dV, dK complete; each MMA warp's last products
  // dP^T of block b issued (barrier b % 4, phase b / 4): the S^T warp follows it
  uint64_t dp_issued[4];
  // tile j's dV, dK staged in its last ring slots: barrier j % 8, phase j / 8. The
  // producer stores up to a ring's depth of tiles late, so one barrier waited on
  // by parity would be ambiguous.
  uint64_t ep_staged[8];
  int item[4];
  int st_bh[8], st_kblk[8], st_last[8];  // producer: tiles by k % 8 (head, key block, last block)
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DkdvBarriers) <= 512, "dK/dV barriers exceed their shared memory");

// TMEM column, relative to the dP^T columns, of the packed bf16 operand for
// k-step kk (16 queries). Warpgroup w holds queries [64 w, 64 w + 64) in
// columns [64 w, 64 w + 64) and finishes them in two halves of 32 queries:
// half h's fp32 dP^T columns [64 w + 32 h, +32) are replaced by its P^T (16
// columns of bf16 pairs) followed by its dS^T (16 columns).
__device__ __forceinline__ uint32_t dkdv_pcol(int kk, bool ds) {
  return (uint32_t)(64 * (kk >> 2) + 32 * ((kk >> 1) & 1) + (ds ? 16 : 0) + 8 * (kk & 1));
}
// k-step of the i-th of the four 16-query steps in query half h: {0, 1, 4, 5} or {2, 3, 6, 7}.
__device__ __forceinline__ constexpr int dkdv_half_kstep(int h, int i) { return 4 * (i >> 1) + 2 * h + (i & 1); }

// A dK/dV tile: (head, key block), its first query block and how many it
// sees, and the sequence's query rows sq and keys sk (padding masks).
struct DkdvTile {
  int bh, kblk, i_start, n, sq, sk;
};

// VARLEN: per-sequence lengths are given (padding masks); without them the
// lengths are the array sizes, which the kernels then take as constants.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ DkdvTile dkdv_tile(int L, const BwdArgs& a, int nkv) {
  DkdvTile t;
  grouped_index(L, a.BH, nkv, a.head_group, t.bh, t.kblk);  // key block 0 (the heaviest) first
  t.sq = a.Nq;
  t.sk = a.Nk;
  if (VARLEN) seq_lens(a.seqlens_q, a.seqlens_k, t.bh / a.H, a.Nq, a.Nk, CAUSAL, t.sq, t.sk);
  if (VARLEN && t.kblk * 128 >= t.sk) {  // padding keys only: one fully masked block gives dk = dv = 0
    t.i_start = 0;
    t.n = 1;
    return t;
  }
  // BQ == BK: query block i sees key block j iff its last row does, 128 i + 127 + sk - sq >= 128 j
  // (with sq = sk: iff i >= j). The last query row sees every key, so n >= 1.
  const int x = t.kblk * 128 - 127 - (t.sk - t.sq);
  t.i_start = CAUSAL && x > 0 ? (x + 127) / 128 : 0;
  t.n = (t.sq + 127) / 128 - t.i_start;
  return t;
}

// DROP: the forward's dropout mask, made again from the seed (philox.cuh).
template <int D, bool CAUSAL, bool VARLEN, bool DROP = false>
__global__ void __launch_bounds__(352, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {  // uniform over the CTA: every thread leaves before any barrier
    if (threadIdx.x == 0) atomicOr(a.status, 16u);
    return;
  }
  DkdvBarriers& bars = *reinterpret_cast<DkdvBarriers*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars.abort;
  float* rowbuf = reinterpret_cast<float*>(smem + C::kOffRow);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Nq = a.Nq;  // rows of the q / lse / D arrays
  const int nkv = (a.Nk + C::BK - 1) / C::BK;
  const int total = a.BH * nkv;

  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int s = 0; s < C::kItemSlots; ++s) {
      mbar_init(&bars.item_full[s], 1);
      mbar_init(&bars.item_empty[s], 2 + 8);  // the two MMA warps and the 8 warpgroup warps
    }
    mbar_init(&bars.k_full, 1);
    mbar_init(&bars.k_empty, 1);
    mbar_init(&bars.v_full, 1);
    mbar_init(&bars.v_empty, 1);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.blk_free[s], 1);
    }
    for (int s = 0; s < C::kDOStages; ++s) mbar_init(&bars.do_full[s], 1);
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, 256);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.ds_half[0], 256);
    mbar_init(&bars.ds_half[1], 256);
    mbar_init(&bars.kv_done, 1);
    for (int j = 0; j < 8; ++j) mbar_init(&bars.ep_staged[j], 256);
    for (int j = 0; j < 4; ++j) mbar_init(&bars.dp_issued[j], 1);
    mbar_init(&bars.teardown, 1);
    mbar_init(&bars.teardown_s, 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  // Tile k of this CTA, as published by the producer in the tile ring; -1 once
  // the counter is exhausted. Every consumer warp reads each slot once and
  // releases it. The wait ignores the abort flag (bounded by time only), so
  // that the warps of a warpgroup agree on their sequence of tiles.
  auto take_tile = [&](int k) -> int {
    const int is = k % C::kItemSlots;
    const bool got = __all_sync(0xffffffffu, mbar_wait_drain(&bars.item_full[is], (k / C::kItemSlots) & 1));
    if (!got) {
      *abort_flag = 1;
      return -1;
    }
    const int L = *reinterpret_cast<volatile int*>(&bars.item[is]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.item_empty[is]);
    return L < total ? L : -1;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // Per tile: K, then Q and dO of each query block in block order (Q first:
    // S^T needs it before dP^T needs dO), with V between Q and dO of the first
    // block. K and V wait for the previous tile's last S^T and dP^T. A ring
    // slot that held a tile's last block holds its staged dV or dK next: the
    // producer stores them (when the slot is about to be reused) and then
    // releases the slots itself. The whole warp waits; one elected lane issues.
    if (elect_one()) {
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_do);
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
    }
    __syncwarp();
    int g = 0, ntiles = 0, next_store = 0;
    int due = INT_MAX;  // last block of tile next_store, once that tile is known
    int q_issued = 0, do_issued = 0, kv_tiles = 0;
    bool ok = true;
    // store tile j's staged dV (dO slot of its last block) and dK (Q slot)
    auto store_tile = [&](int j, bool last) -> bool {
      if (!warp_wait(&bars.ep_staged[j & 7], (j >> 3) & 1, abort_flag)) return false;
      if (elect_one()) {
        const int bh = bars.st_bh[j & 7], kblk = bars.st_kblk[j & 7], gl = bars.st_last[j & 7];
        uint8_t* dv_stage = smem + C::kOffDO + (gl % C::kDOStages) * C::kTileBytes;
        uint8_t* dk_stage = smem + C::kOffQ + (gl % C::kQStages) * C::kTileBytes;
        if (!*abort_flag) {
          for (int pn = 0; pn < D / 64; ++pn) {
            tma_store_3d(&a.tm_dv, dv_stage + pn * kPanelBytes, pn * 64, kblk * C::BK, bh);
            tma_store_3d(&a.tm_dk, dk_stage + pn * kPanelBytes, pn * 64, kblk * C::BK, bh);
          }
          bulk_commit();
        }
        if (last)
          bulk_wait0();
        else
          bulk_wait_read0();
        mbar_arrive(&bars.blk_free[gl % C::kQStages]);  // in place of the MMA warp's release
      }
      __syncwarp();
      return true;
    };
    // before block g reuses a slot of a ring with 'stages' slots
    auto store_due = [&](int g_next, int stages) -> bool {
      while (due <= g_next - stages) {
        if (!store_tile(next_store, false)) return false;
        ++next_store;
        due = next_store < ntiles ? bars.st_last[next_store & 7] : INT_MAX;
      }
      return true;
    };
    for (int k = 0; ok; ++k) {
      const int is = k % C::kItemSlots;
      if (!warp_wait(&bars.item_empty[is], ((k / C::kItemSlots) & 1) ^ 1, abort_flag)) break;
      int L = 0;
      if (lane == 0) {
        L = (int)atomicAdd(&a.work[0], 1u);
        bars.item[is] = L;
      }
      L = __shfl_sync(0xffffffffu, L, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.item_full[is]);  // release: the tile index is visible
      if (L >= total) break;
      const DkdvTile t = dkdv_tile<CAUSAL, VARLEN>(L, a, nkv);
      bars.st_bh[k & 7] = t.bh;  // every lane writes the same values
      bars.st_kblk[k & 7] = t.kblk;
      bars.st_last[k & 7] = g + t.n - 1;
      if (next_store == k) due = g + t.n - 1;
      ntiles = k + 1;
      if (k >= 1 && !(ok = warp_wait(&bars.k_empty, (k - 1) & 1, abort_flag))) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.k_full, C::kTileBytes);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d(smem + C::kOffK + pn * kPanelBytes, &a.tm_k, &bars.k_full, pn * 64, t.kblk * C::BK, t.bh);
      }
      __syncwarp();
      kv_tiles = k + 1;
      for (int it = 0; it < t.n; ++it, ++g) {
        const int qs = g % C::kQStages, ds = g % C::kDOStages;
        if (!(ok = store_due(g, C::kQStages))) break;
        // block g - kQStages used this Q slot (parity 1 of a fresh barrier passes at once)
        if (!(ok = warp_wait(&bars.blk_free[qs], ((g / C::kQStages) & 1) ^ 1, abort_flag))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.q_full[qs], C::kTileBytes);
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(smem + C::kOffQ + qs * C::kTileBytes + pn * kPanelBytes, &a.tm_q, &bars.q_full[qs],
                        pn * 64, (t.i_start + it) * C::BQ, t.bh);
        }
        __syncwarp();
        q_issued = g + 1;
        if (it == 0) {
          if (k >= 1 && !(ok = warp_wait(&bars.v_empty, (k - 1) & 1, abort_flag))) break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&bars.v_full, C::kTileBytes);
            for (int pn = 0; pn < D / 64; ++pn)
              tma_load_3d(smem + C::kOffV + pn * kPanelBytes, &a.tm_v, &bars.v_full, pn * 64, t.kblk * C::BK,
                          t.bh);
          }
          __syncwarp();
        }
        if (!(ok = store_due(g, C::kDOStages))) break;
        // block g - kDOStages used this dO slot (kDOStages <= kQStages: its phase cannot be overtaken)
        if (g >= C::kDOStages) {
          const int b = g - C::kDOStages;
          if (!(ok = warp_wait(&bars.blk_free[b % C::kQStages], (b / C::kQStages) & 1, abort_flag))) break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.do_full[ds], C::kTileBytes);
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(smem + C::kOffDO + ds * C::kTileBytes + pn * kPanelBytes, &a.tm_do, &bars.do_full[ds],
                        pn * 64, (t.i_start + it) * C::BQ, t.bh);
        }
        __syncwarp();
        do_issued = g + 1;
      }
    }
    // the tiles still staged, the last with a full wait; then every copy in flight lands
    while (ok && next_store < ntiles) {
      ok = store_tile(next_store, next_store == ntiles - 1);
      ++next_store;
    }
    if (kv_tiles > 0) {
      mbar_wait_drain(&bars.k_full, (kv_tiles - 1) & 1);
      mbar_wait_drain(&bars.v_full, (kv_tiles - 1) & 1);
    }
    for (int i = max(0, q_issued - C::kQStages); i < q_issued; ++i)
      mbar_wait_drain(&bars.q_full[i % C::kQStages], (i / C::kQStages) & 1);
    for (int i = max(0, do_issued - C::kDOStages); i < do_issued; ++i)
      mbar_wait_drain(&bars.do_full[i % C::kDOStages], (i / C::kDOStages) & 1);
  } else if (warp >= 9) {
    // ------------------------------------------------------------ MMA issuers
    // Each tcgen05 instruction holds its issuing warp about as long as an
    // N = 128 product holds the pipe, so a single issuing warp, with its waits
    // and bookkeeping on top, would leave the pipe idle. Warp 9 issues dK, dV
    // and dP^T, which share TMEM columns and so stay in one thread's issue
    // order; warp 10 issues S^T (columns of its own) once warp 9 has issued the
    // dP^T before it. Each warp stays converged and its operands warp-uniform;
    // one elected lane issues each group of tcgen05 ops.
    {
      constexpr uint32_t kIdKK = idesc_bf16(128, 128, false, false);  // S^T, dP^T: both operands K-major
      constexpr uint32_t kIdTS = idesc_bf16(128, D, false, true);     // dV, dK: A from TMEM, B MN-major
      const uint32_t k_base = smem_u32(smem + C::kOffK), v_base = smem_u32(smem + C::kOffV);
      const uint32_t q_base = smem_u32(smem + C::kOffQ), do_base = smem_u32(smem + C::kOffDO);
      // Descriptors of stage 0; k-steps and other stages add a byte offset / 16 to
      // the start-address field (bits [0,14)).
      const uint64_t dk0 = sdesc_sw128(k_base, 16, 1024), dv0 = sdesc_sw128(v_base, 16, 1024);
      const uint64_t dq0 = sdesc_sw128(q_base, 16, 1024), ddo0 = sdesc_sw128(do_base, 16, 1024);
      const uint64_t dqm0 = sdesc_sw128(q_base, kPanelBytes, 1024), ddom0 = sdesc_sw128(do_base, kPanelBytes, 1024);
      auto koff = [](int kk) -> uint32_t { return ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4; };
      auto q_phase = [&](int g) { return (uint32_t)((g / C::kQStages) & 1); };
      auto do_phase = [&](int g) { return (uint32_t)((g / C::kDOStages) & 1); };
      // Blocks in run order as (position in the tile, tile size, tile index in
      // the run); n == 0 past the end of the run. Each warp walks the run itself.
      struct Blk {
        int it, n, kt;
      };
      Blk cursor = {0, 0, -1};  // the block last handed out
      bool tiles_done = false;
      auto next_blk = [&]() -> Blk {
        if (cursor.it + 1 < cursor.n) {
          ++cursor.it;
          return cursor;
        }
        const int L = tiles_done ? -1 : take_tile(cursor.kt + 1);
        if (L < 0) {
          tiles_done = true;
          return Blk{0, 0, -1};
        }
        cursor = Blk{0, dkdv_tile<CAUSAL, VARLEN>(L, a, nkv).n, cursor.kt + 1};
        return cursor;
      };
      if (warp == 10) {
        // S^T = K Q_g^T of every block, after the warpgroups have read S^T of
        // block g-1 and warp 9 has issued dP^T of block g-1: the pipe then runs
        // it while the warpgroups compute dS^T of block g-1.
        bool ok = true;
        for (int g = 0; ok; ++g) {
          const Blk b = next_blk();
          if (b.n == 0) break;
          const int s = g % C::kQStages;
          if (g == 0)
            ok = warp_wait(&bars.q_full[s], q_phase(g), abort_flag);
          else
            ok = warp_wait2(&bars.s_free, (g - 1) & 1, &bars.q_full[s], q_phase(g), abort_flag) &&
                 warp_wait(&bars.dp_issued[(g - 1) & 3], ((g - 1) >> 2) & 1, abort_flag);
          if (ok && b.it == 0) ok = warp_wait(&bars.k_full, b.kt & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t so = s * C::kTileBytes;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + C::kColS, dk0 + koff(kk), dq0 + koff(kk) + (so >> 4), kIdKK, kk > 0);
            mma_commit(&bars.s_full);
            if (b.it == b.n - 1) mma_commit(&bars.k_empty);  // the tile's last reader of K
          }
          __syncwarp();
        }
        if (elect_one()) mma_commit(&bars.teardown_s);  // the same lane as above: elect.sync picks the lowest
        __syncwarp();
        mbar_wait_drain(&bars.teardown_s, 0);
      } else {
        // dP^T of a tile's first block: it also waits for the tile's V. Other
        // blocks' dP^T is issued with the previous block's second dV/dK half.
        auto issue_dp_first = [&](int g, bool last, int kt) -> bool {  // dP^T = V dO_i^T
          const int s = g % C::kDOStages;
          if (!warp_wait2(&bars.do_full[s], do_phase(g), &bars.v_full, kt & 1, abort_flag)) return false;
          tc_fence_after();
          const uint32_t so = s * C::kTileBytes;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + C::kColDP, dv0 + koff(kk), ddo0 + koff(kk) + (so >> 4), kIdKK, kk > 0);
            mma_commit(&bars.dp_full);
            if (last) mma_commit(&bars.v_empty);  // the tile's last reader of V
            mbar_arrive(&bars.dp_issued[g & 3]);
          }
          __syncwarp();
          return true;
        };
        // Per query block i the critical chain is: the warpgroups' dS^T of
        // block i -> dV and dK of block i -> dP^T of block i+1 (it overwrites
        // the columns that hold P^T and dS^T of block i, so it must follow dK
        // in issue order: the products of one thread execute in that order) ->
        // dS^T of block i+1. dV and dK start on the first half of the queries
        // while the warpgroups still work on the second.
        Blk b0 = next_blk(), b1 = {0, 0, -1};
        bool ok = b0.n > 0;
        if (ok) {
          ok = issue_dp_first(0, b0.n == 1, b0.kt);
          b1 = next_blk();
        }
        for (int g = 0; ok && b0.n > 0; ++g) {
          const int it = b0.it;
          const int qs = g % C::kQStages, ds = g % C::kDOStages;
          const uint32_t qso = qs * C::kTileBytes, dso = ds * C::kTileBytes;
          const bool last = it == b0.n - 1;
          // Within a tile the second half's wait also covers dO of block g+1,
          // and dP^T of block g+1 goes out with that half's products (one
          // elected issue: no commit round trip between them).
          const bool pair_do = !last;
          const bool last1 = b1.it == b1.n - 1;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 1 && pair_do)
              ok = warp_wait2(&bars.ds_half[1], g & 1, &bars.do_full[(g + 1) % C::kDOStages], do_phase(g + 1),
                              abort_flag);
            else
              ok = warp_wait(&bars.ds_half[h], g & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {  // dK += dS^T Q_i
                const int kk = dkdv_half_kstep(h, i);
                mma_ts(tmem + C::kColDK, tmem + C::kColDP + dkdv_pcol(kk, true), dqm0 + ((kk * 2048 + qso) >> 4),
                       kIdTS, (it > 0 || kk > 0) ? 1u : 0u);
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {  // dV += P^T dO_i
                const int kk = dkdv_half_kstep(h, i);
                mma_ts(tmem + C::kColDV, tmem + C::kColDP + dkdv_pcol(kk, false), ddom0 + ((kk * 2048 + dso) >> 4),
                       kIdTS, (it > 0 || kk > 0) ? 1u : 0u);
              }
              if (h == 1) {
                // the block's Q and dO slots are free once dV is done (a tile's last
                // slots are released by the producer once their staged dK, dV are stored)
                mma_commit(last ? &bars.kv_done : &bars.blk_free[qs]);
                if (pair_do) {  // dP^T = V dO_{g+1}^T overwrites P^T, dS^T of block g: it follows dK, dV
                  const uint32_t so1 = ((g + 1) % C::kDOStages) * C::kTileBytes;
#pragma unroll
                  for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tmem + C::kColDP, dv0 + koff(kk), ddo0 + koff(kk) + (so1 >> 4), kIdKK, kk > 0);
                  mma_commit(&bars.dp_full);
                  if (last1) mma_commit(&bars.v_empty);  // the tile's last reader of V
                  mbar_arrive(&bars.dp_issued[(g + 1) & 3]);
                }
              }
            }
            __syncwarp();
          }
          if (!ok) break;
          // a next tile's first block: its dP^T (its S^T comes from warp 10)
          if (b1.n > 0 && !pair_do && !(ok = issue_dp_first(g + 1, last1, b1.kt))) break;
          b0 = b1;
          b1 = b1.n > 0 ? next_blk() : Blk{0, 0, -1};
        }
        if (elect_one()) mma_commit(&bars.teardown);  // the same lane as above: elect.sync picks the lowest
        __syncwarp();
        mbar_wait_drain(&bars.teardown, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int w = warp >> 2;              // columns (queries) [64 w, 64 w + 64) of each block
    const int r = (warp & 3) * 32 + lane;  // key within the block = TMEM lane
    const int tt = threadIdx.x & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS + 64 * w;
    const uint32_t t_dp = tmem + lane_off + C::kColDP + 64 * w;  // dP^T, then P^T | dS^T (bf16)
    const float sl2 = a.scale_log2;
    // Threads 0-63 of the warpgroup fetch lse of the group's 64 queries of
    // query block qb, threads 64-127 fetch D; one block ahead, through
    // registers, and negated (lse also to log2 units) only when stored a block
    // later, so that no thread waits for the load in between.
    auto fetch = [&](const DkdvTile& t, int qb) -> float {
      const int q = qb * C::BQ + 64 * w + (tt & 63);
      const int sq = VARLEN ? t.sq : Nq;
      if (tt < 64) return q < sq ? a.lse[(size_t)t.bh * Nq + q] : INFINITY;  // 2^(x - inf) = 0 past sq
      return q < sq ? a.Dsum[(size_t)t.bh * Nq + q] : 0.f;
    };
    // After a failed wait a warp keeps going without work; at every block the
    // group's named barrier also ANDs the warps' states, so the four warps
    // always agree on their blocks and tiles and meet at the same barriers.
    int L = take_tile(0);
    DkdvTile t = L >= 0 ? dkdv_tile<CAUSAL, VARLEN>(L, a, nkv) : DkdvTile{0, 0, 0, 0, 1, 1};
    float next = L >= 0 ? fetch(t, t.i_start) : 0.f;
    bool ok = L >= 0;
    int g = 0;
    for (int k = 0; L >= 0; ++k) {
      const int key = t.kblk * C::BK + r;
      const int sk = VARLEN ? t.sk : a.Nk;
      const bool key_ok = key < sk;
      const bool keys_all_ok = (t.kblk + 1) * C::BK <= sk;  // uniform over the CTA
      const int off = sk - (VARLEN ? t.sq : Nq);  // causal: query row i sees keys 0 .. i + off
      int L_next = -1;
      DkdvTile nt = {0, 0, 0, 0, 1, 1};
      for (int it = 0; it < t.n; ++it, ++g) {
        const int q0 = (t.i_start + it) * C::BQ;
        float* rb = rowbuf + ((g & 1) * 2 + w) * 128;
        rb[tt] = tt < 64 ? -next * kLog2e : -next;  // -lse (log2 units) | -D
        ok = named_bar_and(1 + w, 128, ok);
        if (it + 1 < t.n) {
          next = fetch(t, t.i_start + it + 1);
        } else {  // the next tile's first block
          L_next = take_tile(k + 1);
          if (L_next >= 0) {
            nt = dkdv_tile<CAUSAL, VARLEN>(L_next, a, nkv);
            next = fetch(nt, nt.i_start);
          }
        }
        if (!ok) continue;
        const float4* rb4 = reinterpret_cast<const float4*>(rb);  // lse at [0, 64), D at [64, 128)
        ok = mbar_wait(&bars.s_full, g & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          continue;
        }
        tc_fence_after();
        uint32_t pk[32];  // P^T row r, queries 64 w .. 64 w + 63, as bf16 pairs
        {
          uint32_t sr[2][32];
          tmem_ld32(t_s, sr[0]);
          tmem_ld32(t_s + 32, sr[1]);
          tmem_ld_wait(sr[0]);
          tmem_ld_wait(sr[1]);
          tc_fence_before();
          mbar_arrive(&bars.s_free);  // S^T is in registers: the next block's S^T may overwrite it
          // Only blocks whose first query row does not see the block's last key
          // (the diagonal, the first block under the causal mask; a second one when
          // sk - sq is not a multiple of 128) and a ragged last key block need
          // masking: there a hidden score becomes -inf, so P = 0 (scale > 0).
          // Query q0 + 64 w + col sees key kblk * BK + r iff q0 + 64 w + col + off >= key.
          if ((CAUSAL && q0 + off < (t.kblk + 1) * C::BK - 1) || !keys_all_ok) {
            const int lim = CAUSAL ? key - off - (q0 + 64 * w) : -1;  // drop columns col < lim
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c < lim || !key_ok) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
          }
          const float2 scale2 = make_float2(sl2, sl2);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const int col = 32 * h + c;  // within the group's 64 queries
              const float4 nl = rb4[col >> 2];  // -lse
              const float2 x01 = ffma2(make_float2(__uint_as_float(sr[h][c]), __uint_as_float(sr[h][c + 1])),
                                       scale2, make_float2(nl.x, nl.y));
              const float2 x23 = ffma2(make_float2(__uint_as_float(sr[h][c + 2]), __uint_as_float(sr[h][c + 3])),
                                       scale2, make_float2(nl.z, nl.w));
              pk[col >> 1] = pack_bf16x2(ex2(x01.x), ex2(x01.y));
              pk[(col >> 1) + 1] = pack_bf16x2(ex2(x23.x), ex2(x23.y));
            }
          }
        }
        // dropout: keep bytes kw[gq], byte b for query q0 + 64 w + 4 gq + b of this thread's key. Each
        // call covers 4 queries x the quad's 4 keys; this lane draws query groups qa, qa + 4, .. and the
        // byte and quad transposes leave it its own key's bytes of all 16 groups.
        uint32_t kw[DROP ? 16 : 1];
        if constexpr (DROP) {
          const uint32_t i4 = (uint32_t)(q0 + 64 * w) >> 2, j4 = (uint32_t)key >> 2, qa = lane & 3;
          const uint32_t thr4 = (uint32_t)a.drop_p256 * 0x01010101u;
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            uint32_t x[4];
            philox::philox4x32_10(j4, i4 + 4 * n + qa, (uint32_t)t.bh, a.drop_offset, a.drop_rk, x);
            philox::byte_transpose(x);  // x[b]: key 4 j4 + b, the group's 4 queries
            philox::quad_transpose(x);  // x[s]: this lane's key, query group 4 n + s
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) kw[4 * n + s4] = philox::keep_bytes(x[s4], thr4);
          }
        }
        ok = mbar_wait(&bars.dp_full, g & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          continue;
        }
        tc_fence_after();
        // Two halves of 32 queries: each replaces its own fp32 dP^T columns by
        // its P^T and dS^T and releases them to the MMA warp at once.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dp[32], dsk[16], pkh[16];
          tmem_ld32(t_dp + 32 * h, dp);
          tmem_ld_wait(dp);
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const int col = 32 * h + c;
            const float4 nd = rb4[16 + (col >> 2)];  // -D
            const uint32_t pa = pk[col >> 1], pb = pk[(col >> 1) + 1];
            const float2 dp01 = make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1]));
            const float2 dp23 = make_float2(__uint_as_float(dp[c + 2]), __uint_as_float(dp[c + 3]));
            float2 e01, e23;  // dP - D, with dropout Z dP - D (Z = 0 or 1 / (1 - p))
            if constexpr (DROP) {
              const uint32_t kc = kw[col >> 2];
              const float f = a.drop_scale;
              e01 = ffma2(dp01, make_float2(philox::keep_factor(kc, 0, f), philox::keep_factor(kc, 1, f)),
                          make_float2(nd.x, nd.y));
              e23 = ffma2(dp23, make_float2(philox::keep_factor(kc, 2, f), philox::keep_factor(kc, 3, f)),
                          make_float2(nd.z, nd.w));
            } else {
              e01 = fadd2(dp01, make_float2(nd.x, nd.y));
              e23 = fadd2(dp23, make_float2(nd.z, nd.w));
            }
            const float2 d01 = fmul2(make_float2(__uint_as_float(pa << 16), __uint_as_float(pa & 0xFFFF0000u)), e01);
            const float2 d23 = fmul2(make_float2(__uint_as_float(pb << 16), __uint_as_float(pb & 0xFFFF0000u)), e23);
            dsk[c >> 1] = pack_bf16x2(d01.x, d01.y);
            dsk[(c >> 1) + 1] = pack_bf16x2(d23.x, d23.y);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pkh[i] = pk[16 * h + i];
            if constexpr (DROP)  // the dropped P^T feeds dV (pair 16 h + i: queries 32 h + 2 i, + 1)
              pkh[i] &= (i & 1) ? philox::pair_mask_hi(kw[(16 * h + i) >> 1]) : philox::pair_mask_lo(kw[(16 * h + i) >> 1]);
          }
          tmem_st16(t_dp + 32 * h, pkh);       // P^T of these queries
          tmem_st16(t_dp + 32 * h + 16, dsk);  // dS^T of these queries
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars.ds_half[h]);
        }
      }
      // Epilogue: warpgroup 0 stages dV in the dO ring slot of the tile's last
      // block, warpgroup 1 stages scale * dK in its Q ring slot; the producer
      // warp stores them. The accumulators may be overwritten by the next
      // tile's first products only after this thread's next ds_half arrival.
      const int g_last = g - 1;
      bool done = ok && mbar_wait(&bars.kv_done, k & 1, abort_flag);
      done = __all_sync(0xffffffffu, done);
      if (done) {
        tc_fence_after();
        uint8_t* stage = w == 0 ? smem + C::kOffDO + (g_last % C::kDOStages) * C::kTileBytes
                                : smem + C::kOffQ + (g_last % C::kQStages) * C::kTileBytes;
        stage_row_bf16<D>(tmem + lane_off + (w == 0 ? C::kColDV : C::kColDK), stage, r, 0,
                          w == 0 ? (DROP ? a.drop_scale : 1.f) : a.scale);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&bars.ep_staged[k & 7]);
      ok = ok && done;
      // the group's warps agree on going on (they read the same tile ring slot)
      if (!named_bar_and(1 + w, 128, L_next >= 0)) break;
      L = L_next;
      t = nt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && bars.abort) atomicOr(a.status, 2u);
}

// ============================================================================ dQ
// Persistent: each CTA takes (head, 128-row query block) tiles from a work
// counter until none is left; within a tile, TMEM lane = query and each
// iteration covers 128 keys. Q is the same for every key block of a tile, so
// the warpgroups copy it into TMEM once and S = Q K^T reads its A operand from
// there. dS has TMEM columns of its own, so S, dP and dQ of consecutive key
// blocks only wait for the warpgroups to have read the previous tile.
//
// Across tiles the pipeline does not drain: K/V rings and the S/dP/dS barriers
// count key blocks over the CTA's whole run, the MMA warp issues S and dP of
// the next tile's first block while the warpgroups write the previous tile's
// dQ, and the next tile's Q is loaded while the current one is processed.
template <int D>
struct DqCfg {
  static constexpr int BQ = 128;  // queries per tile
  static constexpr int BK = 128;  // keys per iteration
  static constexpr int kTileBytes = (D / 64) * kPanelBytes;
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 3;
  static constexpr int kItemSlots = 4;  // tiles fetched ahead by the producer
  // D = 64: an O tile beside dO, from which the warpgroups form D for the tile
  static constexpr bool kFuseD = D == 64;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kOffO = 2 * kTileBytes;  // (kFuseD only)
  static constexpr int kOffK = (kFuseD ? 3 : 2) * kTileBytes;
  static_assert(!kFuseD || kOffO + kTileBytes <= kOffK, "the O tile overlaps the K ring");
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;
  static constexpr uint32_t kColQ = 0;            // Q, bf16 pairs, D / 2 columns
  static constexpr uint32_t kColDS = D / 2;       // dS, bf16 pairs, 64 columns (warpgroup w: [32 w, 32 w + 32))
  static constexpr uint32_t kColS = D / 2 + 64;   // S fp32, 128 columns
  static constexpr uint32_t kColDP = D / 2 + 192;  // dP fp32, 128 columns
  static constexpr uint32_t kColDQ = D / 2 + 320;  // dQ accumulator, D columns
};

struct DqBarriers {
  uint64_t item_full[4], item_empty[4];  // tile ring: producer -> MMA warp and warpgroups
  uint64_t q_full, qt_ready;             // Q buffer (one tile) loaded; Q copied into TMEM
  uint64_t do_full, do_empty;            // dO buffer (one tile; with kFuseD also the O buffer)
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full, s_free, dp_full, dp_free, ds_ready, dq_tile, teardown, teardown_q;
  uint64_t ep_staged, dq_stored;        // dQ of a tile staged in the Q buffer; its store has read it
  int item[4];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqBarriers) <= 512, "dQ barriers exceed their shared memory");

// Copies row r (D bf16) of a 128-row, 128-byte-swizzled tile into TMEM as D / 2
// columns of bf16 pairs at taddr (this thread's lane).
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* tile, int r, uint32_t taddr) {
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    uint32_t v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 x = *reinterpret_cast<const uint4*>(tile + h * kPanelBytes + r * 128 + ((k ^ (r & 7)) << 4));
      v[4 * k] = x.x;
      v[4 * k + 1] = x.y;
      v[4 * k + 2] = x.z;
      v[4 * k + 3] = x.w;
    }
    tmem_st32(taddr + 32 * h, v);
  }
}

// A dQ tile: (head, query block) and the number of key blocks it sees.
// A dQ tile: (head, query block), the key blocks it sees, and the sequence's
// query rows sq and keys sk (padding masks).
struct DqTile {
  int bh, qblk, nk, sq, sk;
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ DqTile dq_tile(int L, const BwdArgs& a, int nq) {
  DqTile t;
  int blk;
  grouped_index(L, a.BH, nq, a.head_group_dq, t.bh, blk);
  t.qblk = CAUSAL ? nq - 1 - blk : blk;  // heaviest first under the causal mask
  t.sq = a.Nq;
  t.sk = a.Nk;
  if (VARLEN) seq_lens(a.seqlens_q, a.seqlens_k, t.bh / a.H, a.Nq, a.Nk, CAUSAL, t.sq, t.sk);
  const int nkv = (t.sk + 127) / 128;
  // BQ == BK: query block i sees key blocks 0 .. (128 i + 127 + sk - sq) / 128 (with sq = sk: 0..i);
  // a block of padding rows only takes one key block, whose P = 0 gives dq = 0
  t.nk = VARLEN && t.qblk * 128 >= t.sq ? 1 : CAUSAL ? min((t.qblk * 128 + 127 + t.sk - t.sq) / 128 + 1, nkv) : nkv;
  return t;
}

template <int D, bool CAUSAL, bool VARLEN, bool DROP = false>
__global__ void __launch_bounds__(352, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DqBarriers& bars = *reinterpret_cast<DqBarriers*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Nq = a.Nq;  // rows of the q / lse / D arrays
  const int nq = (Nq + C::BQ - 1) / C::BQ;
  const int total = a.BH * nq;

  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int s = 0; s < C::kItemSlots; ++s) {
      mbar_init(&bars.item_full[s], 1);
      mbar_init(&bars.item_empty[s], 2 + 8);  // the two MMA warps and the 8 warpgroup warps
    }
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.qt_ready, 256);
    mbar_init(&bars.do_full, 1);
    // the tile's last dP; with kFuseD also every warpgroup thread, once it has formed D
    mbar_init(&bars.do_empty, C::kFuseD ? 1 + 256 : 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, 256);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_free, 256);
    mbar_init(&bars.ds_ready, 256);
    mbar_init(&bars.dq_tile, 1);
    mbar_init(&bars.ep_staged, 256);
    mbar_init(&bars.dq_stored, 1);
    mbar_init(&bars.teardown, 1);
    mbar_init(&bars.teardown_q, 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  // Tile k of this CTA, as published by the producer in the tile ring; -1
  // (and no further tiles) once the counter is exhausted or on abort. Every
  // consumer warp reads each slot once and releases it.
  auto take_tile = [&](int k) -> int {
    const int is = k % C::kItemSlots;
    if (!warp_wait(&bars.item_full[is], (k / C::kItemSlots) & 1, abort_flag)) return -1;
    const int L = *reinterpret_cast<volatile int*>(&bars.item[is]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.item_empty[is]);
    return L < total ? L : -1;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // Per tile: its Q, then K and V of each key block, with dO between K and
    // V of the first block (once the previous tile's last dP has read the dO
    // buffer). The Q buffer is shared with the dQ epilogue: Q of tile k goes
    // in once tile k-1's Q is in TMEM and, from k = 2 on, once the dQ of tile
    // k-2 that the warpgroups staged there has been stored, which this warp
    // does (so that no warpgroup thread waits on a store). The whole warp
    // waits; one elected lane issues.
    if (elect_one()) {
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_do);
    }
    __syncwarp();
    int g = 0;  // key blocks issued over the CTA's run
    int q_loads = 0, do_loads = 0, k_issued = 0, v_issued = 0;
    DqTile hist_even = {}, hist_odd = {};  // the last two tiles (by parity of k), for their dQ stores
    // stores dQ of tile j, staged in the Q buffer, and releases the buffer
    auto store_dq = [&](int j, bool last) -> bool {
      if (!warp_wait(&bars.ep_staged, j & 1, abort_flag)) return false;
      if (elect_one()) {
        if (!*abort_flag) {
          const DqTile tj = (j & 1) ? hist_odd : hist_even;
          for (int pn = 0; pn < D / 64; ++pn)
            tma_store_3d(&a.tm_dq, smem + C::kOffQ + pn * kPanelBytes, pn * 64, tj.qblk * C::BQ, tj.bh);
          bulk_commit();
        }
        if (last)
          bulk_wait0();
        else
          bulk_wait_read0();
        mbar_arrive(&bars.dq_stored);
      }
      __syncwarp();
      return true;
    };
    int ntiles = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int is = k % C::kItemSlots;
      if (!warp_wait(&bars.item_empty[is], ((k / C::kItemSlots) & 1) ^ 1, abort_flag)) break;
      int L = 0;
      if (lane == 0) {
        L = (int)atomicAdd(&a.work[1], 1u);
        bars.item[is] = L;
      }
      L = __shfl_sync(0xffffffffu, L, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.item_full[is]);  // release: the tile index is visible
      if (L >= total) break;
      const DqTile t = dq_tile<CAUSAL, VARLEN>(L, a, nq);
      if (k == 1 && !(ok = warp_wait(&bars.qt_ready, 0, abort_flag))) break;
      if (k >= 2 && !(ok = store_dq(k - 2, false))) break;
      if (k & 1)
        hist_odd = t;
      else
        hist_even = t;
      ntiles = k + 1;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.q_full, C::kTileBytes);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d(smem + C::kOffQ + pn * kPanelBytes, &a.tm_q, &bars.q_full, pn * 64, t.qblk * C::BQ, t.bh);
      }
      __syncwarp();
      q_loads = k + 1;
      for (int j = 0; j < t.nk; ++j, ++g) {
        const int sk = g % C::kKStages, sv = g % C::kVStages;
        if (!(ok = warp_wait(&bars.k_empty[sk], ((g / C::kKStages) & 1) ^ 1, abort_flag))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.k_full[sk], C::kTileBytes);
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(smem + C::kOffK + sk * C::kTileBytes + pn * kPanelBytes, &a.tm_k, &bars.k_full[sk],
                        pn * 64, j * C::BK, t.bh);
        }
        __syncwarp();
        k_issued = g + 1;
        if (j == 0) {
          if (!(ok = warp_wait(&bars.do_empty, (k & 1) ^ 1, abort_flag))) break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&bars.do_full, (C::kFuseD ? 2 : 1) * C::kTileBytes);
            for (int pn = 0; pn < D / 64; ++pn)
              tma_load_3d(smem + C::kOffDO + pn * kPanelBytes, &a.tm_do, &bars.do_full, pn * 64, t.qblk * C::BQ,
                          t.bh);
            if constexpr (C::kFuseD)
              tma_load_3d(smem + C::kOffO, &a.tm_o, &bars.do_full, 0, t.qblk * C::BQ, t.bh);
          }
          __syncwarp();
          do_loads = k + 1;
        }
        if (!(ok = warp_wait(&bars.v_empty[sv], ((g / C::kVStages) & 1) ^ 1, abort_flag))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.v_full[sv], C::kTileBytes);
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(smem + C::kOffV + sv * C::kTileBytes + pn * kPanelBytes, &a.tm_v, &bars.v_full[sv],
                        pn * 64, j * C::BK, t.bh);
        }
        __syncwarp();
        v_issued = g + 1;
      }
    }
    // the last two tiles' dQ, then every copy still in flight lands before the CTA can exit
    if (ok && ntiles >= 2) ok = store_dq(ntiles - 2, false);
    if (ok && ntiles >= 1) ok = store_dq(ntiles - 1, true);
    if (q_loads > 0) mbar_wait_drain(&bars.q_full, (q_loads - 1) & 1);
    if (do_loads > 0) mbar_wait_drain(&bars.do_full, (do_loads - 1) & 1);
    for (int i = max(0, k_issued - C::kKStages); i < k_issued; ++i)
      mbar_wait_drain(&bars.k_full[i % C::kKStages], (i / C::kKStages) & 1);
    for (int i = max(0, v_issued - C::kVStages); i < v_issued; ++i)
      mbar_wait_drain(&bars.v_full[i % C::kVStages], (i / C::kVStages) & 1);
  } else if (warp >= 9) {
    // ------------------------------------------------------------ MMA issuers
    // Two warps share the issue (a tcgen05 instruction holds its warp about as
    // long as an N = 128 product holds the pipe): warp 9 issues S and dP of the
    // next block as soon as the warpgroups have read the current one, warp 10
    // issues dQ += dS K as soon as dS is in TMEM. Their products use disjoint
    // TMEM columns; every hand-over goes through an mbarrier. Each warp stays
    // converged; one elected lane issues each group of tcgen05 ops.
    {
      constexpr uint32_t kIdKK = idesc_bf16(128, 128, false, false);  // S (A from TMEM), dP: B K-major
      constexpr uint32_t kIdTS = idesc_bf16(128, D, false, true);     // dQ: dS from TMEM, K MN-major
      const uint32_t k_base = smem_u32(smem + C::kOffK), v_base = smem_u32(smem + C::kOffV);
      const uint64_t dk0 = sdesc_sw128(k_base, 16, 1024), dv0 = sdesc_sw128(v_base, 16, 1024);
      const uint64_t ddo0 = sdesc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
      const uint64_t dkm0 = sdesc_sw128(k_base, kPanelBytes, 1024);
      auto koff = [](int kk) -> uint32_t { return ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4; };
      auto k_phase = [&](int g) { return (uint32_t)((g / C::kKStages) & 1); };
      auto v_phase = [&](int g) { return (uint32_t)((g / C::kVStages) & 1); };
      if (warp == 10) {
        // dQ += dS K_j of every key block j, once the warpgroups have written dS;
        // the product is K's last reader.
        int k = 0, g = 0;  // tile and key block over the CTA's run
        bool ok = true;
        for (int L = take_tile(0); ok && L >= 0; L = take_tile(++k)) {
          const DqTile t = dq_tile<CAUSAL, VARLEN>(L, a, nq);
          for (int j = 0; j < t.nk; ++j) {
            const int gj = g + j;
            if (!(ok = warp_wait2(&bars.ds_ready, gj & 1, &bars.k_full[gj % C::kKStages], k_phase(gj), abort_flag)))
              break;
            tc_fence_after();
            const uint32_t ko = (uint32_t)((gj % C::kKStages) * C::kTileBytes);
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < C::BK / 16; ++kk)  // dQ += dS K_j  (K = 128 keys)
                mma_ts(tmem + C::kColDQ, tmem + C::kColDS + 32 * (kk >> 2) + 8 * (kk & 3),
                       dkm0 + ((kk * 2048 + ko) >> 4), kIdTS, (j > 0 || kk > 0) ? 1u : 0u);
              mma_commit(&bars.k_empty[gj % C::kKStages]);
              if (j == t.nk - 1) mma_commit(&bars.dq_tile);
            }
            __syncwarp();
          }
          g += t.nk;
        }
        if (elect_one()) mma_commit(&bars.teardown_q);  // the same lane as above: elect.sync picks the lowest
        __syncwarp();
        mbar_wait_drain(&bars.teardown_q, 0);
      } else {
        // S and dP of each key block, once the warpgroups hold the previous
        // block's S (resp. dP) in registers and the operands are loaded.
        auto issue_s = [&](int g) {  // S = Q K_g^T
          const int sk = g % C::kKStages;
          tc_fence_after();
          const uint32_t ko = (uint32_t)(sk * C::kTileBytes) >> 4;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ts(tmem + C::kColS, tmem + C::kColQ + 8 * kk, dk0 + koff(kk) + ko, kIdKK, kk > 0);
            mma_commit(&bars.s_full);
          }
          __syncwarp();
        };
        auto issue_dp = [&](int g, bool last_of_tile) {  // dP = dO V_g^T
          const int sv = g % C::kVStages;
          tc_fence_after();
          const uint32_t vo = (uint32_t)(sv * C::kTileBytes) >> 4;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss(tmem + C::kColDP, ddo0 + koff(kk), dv0 + koff(kk) + vo, kIdKK, kk > 0);
            mma_commit(&bars.dp_full);
            mma_commit(&bars.v_empty[sv]);
            if (last_of_tile) mma_commit(&bars.do_empty);  // the tile's last reader of dO
          }
          __syncwarp();
        };
        int k = 0, g = 0;  // tile and key block over the CTA's run
        int L = take_tile(0);
        DqTile t = L >= 0 ? dq_tile<CAUSAL, VARLEN>(L, a, nq) : DqTile{0, 0, 0, 1, 1};
        bool ok = L >= 0;
        while (ok) {
          // the tile's first block: S needs its Q in TMEM (the warpgroups copy it
          // after the previous tile's last S has been read), dP its dO (loaded
          // once the previous tile's last dP has read the buffer)
          if (!(ok = (g == 0 ? warp_wait(&bars.qt_ready, k & 1, abort_flag)
                             : warp_wait2(&bars.s_free, (g - 1) & 1, &bars.qt_ready, k & 1, abort_flag)) &&
                     warp_wait(&bars.k_full[g % C::kKStages], k_phase(g), abort_flag)))
            break;
          issue_s(g);
          if (!(ok = (g == 0 ? warp_wait(&bars.do_full, k & 1, abort_flag)
                             : warp_wait2(&bars.dp_free, (g - 1) & 1, &bars.do_full, k & 1, abort_flag)) &&
                     warp_wait(&bars.v_full[g % C::kVStages], v_phase(g), abort_flag)))
            break;
          issue_dp(g, t.nk == 1);
          for (int j = 1; j < t.nk; ++j) {
            const int gj = g + j;
            if (!(ok = warp_wait2(&bars.s_free, (gj - 1) & 1, &bars.k_full[gj % C::kKStages], k_phase(gj),
                                  abort_flag)))
              break;
            issue_s(gj);
            if (!(ok = warp_wait2(&bars.dp_free, (gj - 1) & 1, &bars.v_full[gj % C::kVStages], v_phase(gj),
                                  abort_flag)))
              break;
            issue_dp(gj, j == t.nk - 1);
          }
          if (!ok) break;
          g += t.nk;
          ++k;
          if ((L = take_tile(k)) < 0) break;
          t = dq_tile<CAUSAL, VARLEN>(L, a, nq);
        }
        if (elect_one()) mma_commit(&bars.teardown);  // the same lane as above: elect.sync picks the lowest
        __syncwarp();
        mbar_wait_drain(&bars.teardown, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int w = warp >> 2;              // key columns [64 w, 64 w + 64) of each block
    const int r = (warp & 3) * 32 + lane;  // query within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    const uint32_t t_s = tmem + lane_off + C::kColS + 64 * w;
    const uint32_t t_dp = tmem + lane_off + C::kColDP + 64 * w;
    const uint32_t t_ds = tmem + lane_off + C::kColDS + 32 * w;
    // this thread's row terms for a tile, loaded early and converted when
    // the tile starts (rows past sq get P = 0 then; rows past Nq read row Nq - 1)
    auto load_row_terms = [&](const DqTile& t, float& lse_raw, float& d_raw) {
      const int q = min(t.qblk * C::BQ + r, Nq - 1);
      lse_raw = a.lse[(size_t)t.bh * Nq + q];
      d_raw = C::kFuseD ? 0.f : a.Dsum[(size_t)t.bh * Nq + q];  // (formed in the tile's first block)
    };
    auto row_terms = [&](const DqTile& t, float lse_raw, float d_raw, float& lse2, float& dsum) {
      const bool in = t.qblk * C::BQ + r < (VARLEN ? t.sq : Nq);
      lse2 = in ? lse_raw * kLog2e : INFINITY;
      dsum = in ? d_raw : 0.f;
    };
    // Q of tile k into TMEM (row r = lane r): warpgroup w copies the 64-column
    // panel w. The Q buffer is released separately: after the first tile's
    // copy at once, later it first stages the previous tile's dQ.
    auto copy_q = [&](int k) -> bool {
      bool ok = mbar_wait(&bars.q_full, k & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok && w < D / 64) {
        tile_row_to_tmem<64>(smem + C::kOffQ + w * kPanelBytes, r, tmem + lane_off + C::kColQ + 32 * w);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bars.qt_ready);
      return ok;
    };
    int k = 0, g = 0;
    int L = take_tile(0);
    bool ok = L >= 0;
    DqTile t = ok ? dq_tile<CAUSAL, VARLEN>(L, a, nq) : DqTile{0, 0, 0, 1, 1};
    float lse2 = 0.f, dsum = 0.f;
    if (ok) {
      float lr, dr;
      load_row_terms(t, lr, dr);
      row_terms(t, lr, dr, lse2, dsum);
      ok = copy_q(0);
    }
    while (ok) {
      const int q = t.qblk * C::BQ + r;
      if constexpr (C::kFuseD) {
        // D of this thread's row, dO . O over the row's 64 features (every
        // warpgroup thread forms its row's D; warpgroup 0 also writes it for the
        // dK/dV kernel), then the dO and O tiles are released to the producer
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.do_full, k & 1, abort_flag));
        if (!ok) break;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int off = r * 128 + ((c ^ (r & 7)) << 4);  // 16-byte chunk c of the 128-byte-swizzled row
          const uint4 x = *reinterpret_cast<const uint4*>(smem + C::kOffDO + off);
          const uint4 y = *reinterpret_cast<const uint4*>(smem + C::kOffO + off);
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc0 = fmaf(__uint_as_float(xs[i] << 16), __uint_as_float(ys[i] << 16), acc0);
            acc1 = fmaf(__uint_as_float(xs[i] & 0xFFFF0000u), __uint_as_float(ys[i] & 0xFFFF0000u), acc1);
          }
        }
        mbar_arrive(&bars.do_empty);
        const float drow = acc0 + acc1;
        if (w == 0 && q < Nq) a.Dsum[(size_t)t.bh * Nq + q] = drow;
        dsum = q < (VARLEN ? t.sq : Nq) ? drow : 0.f;
      }
      for (int j = 0; j < t.nk; ++j) {
        const int gj = g + j;
        ok = mbar_wait(&bars.s_full, gj & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int k0 = j * C::BK + 64 * w;  // first key of this warpgroup's columns
        float2 pf[32];  // P, this thread's row, keys k0 .. k0 + 63 (fp32: only dS, not P, feeds a product here)
        {
          uint32_t sr[2][32];
          tmem_ld32(t_s, sr[0]);
          tmem_ld32(t_s + 32, sr[1]);
          tmem_ld_wait(sr[0]);
          tmem_ld_wait(sr[1]);
          tc_fence_before();
          mbar_arrive(&bars.s_free);  // S is in registers: the next block's S may overwrite it
          // Only blocks reaching past the tile's first row's last key (the diagonal,
          // or two blocks when sk - sq is not a multiple of 128) and a ragged last
          // key block need masking: keys past the causal limit or past sk get a
          // -inf score, so P = 0 (scale > 0).
          const int sk = VARLEN ? t.sk : a.Nk;
          const int off = sk - (VARLEN ? t.sq : Nq);  // causal: query row i sees keys 0 .. i + off
          if ((CAUSAL && (j + 1) * C::BK - 1 > t.qblk * C::BQ + off) || (j + 1) * C::BK > sk) {
            const int lim = (CAUSAL ? min(q + off, sk - 1) : sk - 1) - k0;  // keep key k0 + col iff col <= lim
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c > lim) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
          }
          const float2 scale2 = make_float2(sl2, sl2), shift2 = make_float2(-lse2, -lse2);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 x =
                  ffma2(make_float2(__uint_as_float(sr[h][c]), __uint_as_float(sr[h][c + 1])), scale2, shift2);
              pf[(32 * h + c) >> 1] = make_float2(ex2(x.x), ex2(x.y));
            }
          }
        }
        // dropout: keep bytes kw[gk], byte b for key k0 + 4 gk + b of this thread's query. This lane
        // draws key groups qa, qa + 4, .. for the quad's 4 queries; the quad exchange leaves it its row's.
        uint32_t kw[DROP ? 16 : 1];
        if constexpr (DROP) {
          const uint32_t j4 = (uint32_t)k0 >> 2, i4 = (uint32_t)q >> 2, qa = lane & 3;
          const uint32_t thr4 = (uint32_t)a.drop_p256 * 0x01010101u;
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            uint32_t x[4];
            philox::philox4x32_10(j4 + 4 * n + qa, i4, (uint32_t)t.bh, a.drop_offset, a.drop_rk, x);
            philox::quad_transpose(x);  // x[s]: this lane's query, key group 4 n + s
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) kw[4 * n + s4] = philox::keep_bytes(x[s4], thr4);
          }
        }
        ok = mbar_wait(&bars.dp_full, gj & 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t dp[2][32], dsk[32];
        tmem_ld32(t_dp, dp[0]);
        tmem_ld32(t_dp + 32, dp[1]);
        tmem_ld_wait(dp[0]);
        tmem_ld_wait(dp[1]);
        tc_fence_before();
        mbar_arrive(&bars.dp_free);  // dP is in registers: the next block's dP may overwrite it
        const float2 nd2 = make_float2(-dsum, -dsum);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int col = 32 * h + c;
            // dS = P (dP - D), with dropout P (Z dP - D)
            const float2 dpc = make_float2(__uint_as_float(dp[h][c]), __uint_as_float(dp[h][c + 1]));
            float2 e;
            if constexpr (DROP) {
              const uint32_t kc = kw[col >> 2];
              const int b = col & 3;
              e = ffma2(dpc, make_float2(philox::keep_factor(kc, b, a.drop_scale), philox::keep_factor(kc, b + 1, a.drop_scale)),
                        nd2);
            } else {
              e = fadd2(dpc, nd2);
            }
            const float2 d = fmul2(pf[col >> 1], e);
            dsk[col >> 1] = pack_bf16x2(d.x, d.y);
          }
        }
        if (gj > 0) {
          // The dQ product of the previous key block has read its dS: the commit
          // that releases that block's K ring slot follows it. It is the
          // (gj-1) / kKStages-th use of the slot, and the slot cannot be reused
          // before this thread has stored dS of this block (the next product
          // on it needs this dS).
          ok = mbar_wait(&bars.k_empty[(gj - 1) % C::kKStages], ((gj - 1) / C::kKStages) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st32(t_ds, dsk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.ds_ready);
      }
      if (!ok) break;
      // The next tile's Q goes into TMEM now (this tile's last S has been read),
      // so that its first S runs while this tile's dQ is written out; its row
      // terms are loaded here and converted when it starts.
      g += t.nk;
      L = take_tile(k + 1);
      DqTile nt = {0, 0, 0};
      float lse_next = 0.f, d_next = 0.f;
      if (L >= 0) {
        nt = dq_tile<CAUSAL, VARLEN>(L, a, nq);
        load_row_terms(nt, lse_next, d_next);
        ok = copy_q(k + 1);
      }
      // Epilogue of the finished tile: dq = bf16(scale * dQ), staged row by row
      // in the Q buffer for the producer warp to store; warpgroup w converts
      // features [D/2 w, D/2 w + D/2). The buffer must hold nothing the
      // producer still needs: the next tile's Q has been copied out by every
      // thread, and the previous tile's dQ has been read by its store.
      bool done = mbar_wait(&bars.dq_tile, k & 1, abort_flag);
      if (L >= 0) done = done && mbar_wait(&bars.qt_ready, (k + 1) & 1, abort_flag);
      if (k >= 1) done = done && mbar_wait(&bars.dq_stored, (k - 1) & 1, abort_flag);
      done = __all_sync(0xffffffffu, done);
      if (done) {
        tc_fence_after();
        stage_row_bf16<D / 2>(tmem + lane_off + C::kColDQ + (D / 2) * w, smem + C::kOffQ, r, (D / 2) * w, a.scale);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&bars.ep_staged);
      ok = ok && done;
      if (L < 0) break;
      t = nt;
      row_terms(t, lse_next, d_next, lse2, dsum);
      ++k;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && bars.abort) atomicOr(a.status, 4u);
}

// ============================================================================ D = rowsum(dO o O)
// Each thread handles 8 consecutive elements of one row; D / 8 threads share a row.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int kThreadsPerRow = D / 8;
  const long long rows = (long long)a.BH * a.Nq;
  const long long row = (long long)blockIdx.x * (256 / kThreadsPerRow) + threadIdx.x / kThreadsPerRow;
  const int part = threadIdx.x % kThreadsPerRow;
  float acc = 0.f;
  if (row < rows) {
    const uint4 ov = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.o) + row * D + part * 8);
    const uint4 gv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.dO) + row * D + part * 8);
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(gw[i] << 16), acc);
      acc = fmaf(__uint_as_float(ow[i] & 0xFFFF0000u), __uint_as_float(gw[i] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int off = kThreadsPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) a.Dsum[row] = acc;
  if (blockIdx.x == 0 && threadIdx.x < 2) a.work[threadIdx.x] = 0u;  // tile counters of the next two kernels
  // one thread per sequence checks its lengths (the other kernels clamp them)
  const long long seq_rows = (long long)a.H * a.Nq;
  if ((a.seqlens_q || a.seqlens_k) && part == 0 && row < rows && row % seq_rows == 0) {
    int sq, sk;
    if (seq_lens(a.seqlens_q, a.seqlens_k, (int)(row / seq_rows), a.Nq, a.Nk, a.causal != 0, sq, sk))
      atomicOr(a.status, kStatusBadLength);
  }
}

// The d = 64 backward's first kernel (its dQ kernel forms D): the work counters
// of the two main kernels are reset, and one thread per sequence checks its lengths.
__global__ void __launch_bounds__(32) fa_bwd_start_kernel(const __grid_constant__ BwdArgs a) {
  if (threadIdx.x < 2) a.work[threadIdx.x] = 0u;
  if (a.seqlens_q || a.seqlens_k)
    for (int b = (int)threadIdx.x; b < a.BH / a.H; b += 32) {
      int sq, sk;
      if (seq_lens(a.seqlens_q, a.seqlens_k, b, a.Nq, a.Nk, a.causal != 0, sq, sk)) atomicOr(a.status, kStatusBadLength);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_t(const BwdArgs& a, int num_sms, cudaStream_t stream) {
  cudaError_t e;
  const bool varlen = a.seqlens_q || a.seqlens_k;
  auto kv = varlen ? fa_bwd_dkdv_kernel<D, CAUSAL, true> : fa_bwd_dkdv_kernel<D, CAUSAL, false>;
  if (a.drop_p256 > 0) kv = fa_bwd_dkdv_kernel<D, CAUSAL, false, true>;  // dropout: no lengths
  auto kq = varlen ? fa_bwd_dq_kernel<D, CAUSAL, true> : fa_bwd_dq_kernel<D, CAUSAL, false>;
  if (a.drop_p256 > 0) kq = fa_bwd_dq_kernel<D, CAUSAL, false, true>;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvCfg<D>::kSmemBytes)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmemBytes)) !=
      cudaSuccess)
    return e;
  // persistent: one CTA per SM at most (both main kernels take their tiles from counters)
  const long long kv_tiles = (long long)a.BH * ((a.Nk + 127) / 128), q_tiles = (long long)a.BH * ((a.Nq + 127) / 128);
  const unsigned kv_ctas = (unsigned)std::min<long long>(kv_tiles, num_sms);
  const unsigned q_ctas = (unsigned)std::min<long long>(q_tiles, num_sms);
  if constexpr (DqCfg<D>::kFuseD) {
    // the dQ kernel forms D and writes it; the dK/dV kernel reads it after
    fa_bwd_start_kernel<<<1, 32, 0, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kq<<<q_ctas, 352, DqCfg<D>::kSmemBytes, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kv<<<kv_ctas, 352, DkdvCfg<D>::kSmemBytes, stream>>>(a);
  } else {
    const long long rows = (long long)a.BH * a.Nq;
    const int rows_per_block = 256 / (D / 8);
    fa_bwd_prep_kernel<D><<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), 256, 0, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kv<<<kv_ctas, 352, DkdvCfg<D>::kSmemBytes, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kq<<<q_ctas, 352, DqCfg<D>::kSmemBytes, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& args, int num_sms, cudaStream_t stream) {
  BwdArgs a = args;
  // a CTA's fixed cost (loads before the first product, epilogue) is about 2.5 blocks of work
  a.head_group = pick_head_group(a.BH, (a.Nk + 127) / 128, a.causal != 0, num_sms, 2.5);
  a.head_group_dq = pick_head_group(a.BH, (a.Nq + 127) / 128, a.causal != 0, num_sms, 2.5);
  if (a.d == 64)
    return a.causal ? launch_bwd_t<64, true>(a, num_sms, stream) : launch_bwd_t<64, false>(a, num_sms, stream);
  return a.causal ? launch_bwd_t<128, true>(a, num_sms, stream) : launch_bwd_t<128, false>(a, num_sms, stream);
}

}  // namespace fa
