// Forward pass of exact attention on sm_103a.
//
// One CTA owns two 128-row query tiles of one (batch, head) (one tile at
// d = 64, where two CTAs share an SM) and streams the head's key/value blocks
// (128 rows each) past them, as in the blocked loop of
// "FlashAttention and GPU Memory", chapter 07 (a query block stays on the SM
// while the key and value blocks stream through; of all the results, only O
// goes back to device memory). Per key block and query tile:
//   S = Q K^T                 tcgen05.mma, bf16 operands from shared memory,
//                             fp32 accumulator in tensor memory (TMEM)
//   m, l, P                   running row max / sum of exponentials (chapter
//                             08), one TMEM lane (= one query row) per thread,
//                             exponentials in base 2 with the scale folded in
//   O += P V                  tcgen05.mma, P read back from TMEM as bf16
// and at the end O / l and the row logsumexp are written.
//
// Warp roles (320 threads with two tiles): warps 0-3 and 4-7 are the
// softmax/epilogue warpgroups of query tiles 0 and 1, warp 8 issues TMA loads,
// warp 9 issues the MMAs and owns the TMEM allocation (with one tile: warps
// 0-3, 4 and 5). The tiles alternate on the tensor core, within a CTA or
// between the two CTAs of an SM, so that one tile's softmax overlaps the other
// tile's products (the staggering the pages describe for the third version,
// chapter 11).
//
// Template flags add the other variants without changing this one: per-
// sequence lengths (padding masks), E4M3 inputs with 8-bit products, and
// dropout of P with a Philox mask.
//
// The running maximum used as the exponent reference is only moved when the
// true row maximum exceeds it by more than 2^8; O and l are always scaled
// against the same reference, so the final O / l is unchanged in exact
// arithmetic while most O rescales are skipped.
#include "fa_internal.h"
#include "block_order.cuh"
#include "philox.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace fa::ptx;

constexpr float kLn2 = 0.693147180559945309417f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// 8-bit P: the reference is an integer and P = 2^(x - m_ref + kP8Bias) with
// x <= m_ref + kP8Lag, so P <= 2^8 (E4M3 holds up to 448) and rounding P at
// any reference gives the same values up to a power of two.
constexpr float kP8Bias = 6.0f;
constexpr float kP8Lag = 2.0f;

// FP8: q, k, v are E4M3 (one byte per element) and both products use 8-bit
// operands (P is rounded to E4M3); o stays bf16.
template <int D, bool FP8 = false>
struct FwdCfg {
  static constexpr int BM = 128;                 // query rows per tile = TMEM lanes
  static constexpr int BN = 128;                 // keys per block
  static constexpr int kElem = FP8 ? 1 : 2;      // bytes per input element
  static constexpr int kPanels = D * kElem / 128;  // 128-byte-wide column panels per input row
  static constexpr int kPanelBytes = 128 * 128;  // 128 rows x 128 bytes
  static constexpr int kTileBytes = kPanels * kPanelBytes;
  static constexpr int kOPanels = D / 64;        // panels of a bf16 output row
  // a query tile's slot also stages that tile's bf16 O for the store
  static constexpr int kQSlotBytes = (kPanels > kOPanels ? kPanels : kOPanels) * kPanelBytes;
  static constexpr int kKStep = FP8 ? 32 : 16;   // K of one MMA instruction
  // Query tiles per CTA. At d = 64 a CTA takes one tile (256 TMEM columns,
  // under 113 KB of shared memory), so that two CTAs share an SM and one's
  // loads and epilogue overlap the other's main loop; otherwise two tiles.
  static constexpr int kTiles = D == 64 ? 1 : 2;
  static constexpr int kCtasPerSm = 3 - kTiles;
  static constexpr int kRows = 128 * kTiles;      // query rows per CTA
  static constexpr uint32_t kTmemCols = kTiles == 2 ? 512u : 256u;
  // K of a block is released once both tiles' S have read it, V only once both
  // PV products have: V gets the deeper ring, so its load has more than one
  // block's time to land.
  static constexpr int kKStages = FP8 ? 4 : 2;
  static constexpr int kVStages = FP8 ? 4 : 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTiles * kQSlotBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
  static_assert(kCtasPerSm == 1 || 2 * (kSmemBytes + 1024) <= 233472, "two CTAs must fit an SM's shared memory");
  // TMEM columns: S_t (fp32, 128 columns; P_t as bf16 reuses its first 64,
  // as E4M3 its first 32) and O_t (fp32, D columns) for query tiles t = 0, 1.
  __host__ __device__ static constexpr uint32_t col_s(int t) { return (uint32_t)t * 128u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 128u * kTiles + (uint32_t)t * D; }
  // a softmax warpgroup per tile, then the TMA warp and the MMA warp
  static constexpr int kThreads = 128 * kTiles + 64;
  static constexpr int kWarpTma = 4 * kTiles, kWarpMma = 4 * kTiles + 1;
};

struct FwdBarriers {
  uint64_t q_full[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t teardown;
  uint32_t tmem_base;
  int abort;
};

// o = 0 and lse = -inf for rows [r0, r0 + n) of head bh (padding rows that
// no product touches), by threads tid of nthr with plain 16-byte stores.
template <int D>
__device__ inline void zero_rows(const FwdArgs& a, int bh, int r0, int n, int tid, int nthr) {
  constexpr int kChunks = D / 8;  // 16-byte chunks of a bf16 row
  uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.o) + ((size_t)bh * a.Nq + r0) * D * 2);
  for (int i = tid; i < n * kChunks; i += nthr) o[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < n; i += nthr) a.lse[(size_t)bh * a.Nq + r0 + i] = -INFINITY;
}

// VARLEN: per-sequence lengths are given (padding masks); without them the
// lengths are the array sizes, which the kernel then takes as constants.
// FP8: E4M3 inputs and 8-bit products (FwdCfg). DROP: dropout of P after the
// softmax with a Philox mask (philox.cuh); O / l takes the 1 / (1 - p) factor.
template <int D, bool CAUSAL, bool VARLEN, bool FP8 = false, bool DROP = false>
__global__ void __launch_bounds__(FwdCfg<D, FP8>::kThreads, FwdCfg<D, FP8>::kCtasPerSm)
    fa_fwd_kernel(const __grid_constant__ FwdArgs a) {
  using C = FwdCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBarriers& bars = *reinterpret_cast<FwdBarriers*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Nq = a.Nq;  // rows of the q / o / lse arrays
  // grid.x runs over (head, query block) pairs, so the number of query blocks
  // is not bound by the 65535 limit of grid.y
  const int nqblk = (Nq + C::kRows - 1) / C::kRows;
  int bh, blk;
  grouped_index((int)blockIdx.x, a.BH, nqblk, a.head_group, bh, blk);
  const int qblk = CAUSAL ? nqblk - 1 - blk : blk;  // heaviest first under the causal mask
  // this sequence's query rows sq and keys sk (all of them without padding masks)
  int sq = Nq, sk = a.Nk;
  if (VARLEN && seq_lens(a.seqlens_q, a.seqlens_k, bh / a.H, Nq, a.Nk, CAUSAL, sq, sk) && threadIdx.x == 0)
    atomicOr(a.status, kStatusBadLength);
  const int off = sk - sq;  // causal: query row i sees keys 0 .. i + off
  const int nkv = (sk + C::BN - 1) / C::BN;
  // this CTA's key blocks: [jb, je) (all of them unless the keys are split)
  const int jb = (int)blockIdx.z * a.split_blocks;
  const int je = min(nkv, jb + a.split_blocks);
  int nb[2];  // key blocks each query tile sees in the range, from jb on (none for an absent tile)
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = qblk * C::kRows + t * 128;
    const int last_key = CAUSAL ? min(min(r0 + 127, sq - 1) + off, sk - 1) : sk - 1;
    nb[t] = t < C::kTiles && r0 < sq ? max(0, min(last_key / C::BN + 1, je) - jb) : 0;
  }
  const int nb_max = max(nb[0], nb[1]);
  if (nb_max == 0) {
    // No row of this CTA sees a key of its range: either the keys are split
    // and the range has no weight in the merge, or every row is padding
    // (o = 0, lse = -inf). The condition is uniform over the CTA, so every
    // thread leaves before any barrier.
    if (a.n_split > 1) {
      if ((int)threadIdx.x < C::kRows) {
        const int row = qblk * C::kRows + (int)threadIdx.x;
        if (row < Nq) a.lse_part[((size_t)blockIdx.z * a.BH + bh) * Nq + row] = -INFINITY;
      }
    } else if (VARLEN) {
      const int r0 = qblk * C::kRows;
      zero_rows<D>(a, bh, r0, min(C::kRows, Nq - r0), (int)threadIdx.x, (int)blockDim.x);
    }
    return;
  }

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.q_full[0], 1);
    mbar_init(&bars.q_full[1], 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], 128);
      mbar_init(&bars.o_done[t], 1);
    }
    mbar_init(&bars.teardown, 1);
    fence_mbar_init();
  }
  if (warp == C::kWarpMma) {
    tmem_alloc(&bars.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;

  if (warp == C::kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    // Q tile 0, then K and V of each key block, with Q tile 1 between K and
    // V of the first block (the first S needs Q tile 0 and K only). The whole
    // warp waits on the ring barriers; one elected lane issues.
    auto load_q = [&](int t) {
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.q_full[t], C::kTileBytes);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_3d(smem + C::kOffQ + t * C::kQSlotBytes + pn * C::kPanelBytes, &a.tm_q, &bars.q_full[t],
                      pn * (128 / C::kElem),
                      qblk * C::kRows + t * 128, bh);
      }
      __syncwarp();
    };
    if (elect_one()) {
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
    }
    __syncwarp();
    // test hook: without the first Q tile, the MMA warp's first wait expires
    const bool q0_issued = a.test_fault != 1;
    if (q0_issued) load_q(0);
    bool q1_issued = false;
    int nk_issued = 0, nv_issued = 0;
    for (int j = 0; j < nb_max; ++j) {
      const int sk = j % C::kKStages, sv = j % C::kVStages;
      if (!warp_wait(&bars.k_empty[sk], ((j / C::kKStages) & 1) ^ 1, abort_flag)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.k_full[sk], C::kTileBytes);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_3d(smem + C::kOffK + sk * C::kTileBytes + pn * C::kPanelBytes, &a.tm_k, &bars.k_full[sk],
                      pn * (128 / C::kElem), (jb + j) * C::BN, bh);
      }
      __syncwarp();
      nk_issued = j + 1;
      if (C::kTiles == 2 && j == 0) {
        load_q(1);
        q1_issued = true;
      }
      if (!warp_wait(&bars.v_empty[sv], ((j / C::kVStages) & 1) ^ 1, abort_flag)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.v_full[sv], C::kTileBytes);
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_3d(smem + C::kOffV + sv * C::kTileBytes + pn * C::kPanelBytes, &a.tm_v, &bars.v_full[sv],
                      pn * (128 / C::kElem), (jb + j) * C::BN, bh);
      }
      __syncwarp();
      nv_issued = j + 1;
    }
    // Let every issued copy land before the CTA can exit.
    if (q0_issued) mbar_wait_drain(&bars.q_full[0], 0);
    if (q1_issued) mbar_wait_drain(&bars.q_full[1], 0);
    for (int i = max(0, nk_issued - C::kKStages); i < nk_issued; ++i)
      mbar_wait_drain(&bars.k_full[i % C::kKStages], (i / C::kKStages) & 1);
    for (int i = max(0, nv_issued - C::kVStages); i < nv_issued; ++i)
      mbar_wait_drain(&bars.v_full[i % C::kVStages], (i / C::kVStages) & 1);
  } else if (warp == C::kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp follows the schedule, so it stays converged and its
    // operands warp-uniform; one elected lane issues each group of tcgen05
    // ops (elect.sync picks the lowest active lane, so always the same one,
    // which matters because a commit tracks the issuing thread's MMAs).
    {
      // Q, K both K-major; P from TMEM, V MN-major
      constexpr uint32_t kIdS = FP8 ? idesc_e4m3(128, C::BN, false, false) : idesc_bf16(128, C::BN, false, false);
      constexpr uint32_t kIdO = FP8 ? idesc_e4m3(128, D, false, true) : idesc_bf16(128, D, false, true);
      const uint32_t q_base = smem_u32(smem + C::kOffQ);
      const uint32_t k_base = smem_u32(smem + C::kOffK);
      const uint32_t v_base = smem_u32(smem + C::kOffV);
      // Descriptors of Q tile 0 and K/V stage 0. Other k-steps, tiles and stages
      // add a byte offset / 16 to the start-address field (bits [0,14)).
      const uint64_t dq0 = sdesc_sw128(q_base, 16, 1024), dk0 = sdesc_sw128(k_base, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(v_base, C::kPanelBytes, 1024);
      auto issue_s = [&](int t, int st) {  // by the elected lane
        const uint32_t d_s = tmem + C::col_s(t);
        const uint32_t qo = (uint32_t)(t * C::kQSlotBytes) >> 4, ko = (uint32_t)(st * C::kTileBytes) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / C::kKStep; ++kk) {  // each k-step reads 32 bytes of every row
          const uint32_t off = ((kk >> 2) * C::kPanelBytes + (kk & 3) * 32) >> 4;
          if constexpr (FP8)
            mma_ss_f8(d_s, dq0 + qo + off, dk0 + ko + off, kIdS, kk > 0);
          else
            mma_ss(d_s, dq0 + qo + off, dk0 + ko + off, kIdS, kk > 0);
        }
        mma_commit(&bars.s_full[t]);
      };
      bool ok = warp_wait(&bars.q_full[0], 0, abort_flag) && warp_wait(&bars.k_full[0], 0, abort_flag);
      if (ok) {
        tc_fence_after();
        if (elect_one() && nb[0] > 0) issue_s(0, 0);
        __syncwarp();
        if (C::kTiles == 2) ok = warp_wait(&bars.q_full[1], 0, abort_flag);
      }
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
          if (C::kTiles == 2 && nb[1] > 0) issue_s(1, 0);
          mma_commit(&bars.k_empty[0]);
        }
        __syncwarp();
      }
      // Per key block j and tile t: O_t += P_t V_j, then at once S_t for block
      // j + 1. S_t(j + 1) overwrites the columns P_t(j) occupies; the products
      // of one thread execute in issue order, so PV_t(j) has read P_t(j)
      // before S_t(j + 1) writes them, and when S_t(j + 1) completes, so has
      // PV_t(j) (the softmax may then rescale O_t).
      for (int j = 0; ok && j < nb_max; ++j) {
        const int s = j % C::kVStages;
        const uint32_t ph = (j / C::kVStages) & 1;
        const int v_last = j < nb[1] ? 1 : 0;  // the tile whose PV reads V_j last
        const int jn = j + 1, sn = jn % C::kKStages;
        const bool k_next = jn < nb_max;  // some tile reads K of the next block
        // V of this block, tile 0's P and the next block's K (loaded two blocks
        // ahead, so nearly always there) in one wait: each mbarrier probe costs
        // about a hundred cycles, and the three overlap.
        ok = warp_wait3(&bars.v_full[s], ph, j < nb[0] ? &bars.p_full[0] : &bars.v_full[s], j < nb[0] ? (j & 1) : ph,
                        k_next ? &bars.k_full[sn] : &bars.v_full[s], k_next ? (jn / C::kKStages) & 1 : ph, abort_flag);
        if (!ok) break;
        for (int t = 0; t < C::kTiles && ok; ++t) {
          if (j < nb[t]) {
            if (t == 1 && !(ok = warp_wait(&bars.p_full[t], j & 1, abort_flag))) break;
            tc_fence_after();
            if (elect_one()) {
              const uint32_t a_p = tmem + C::col_s(t);
              const uint32_t d_o = tmem + C::col_o(t);
              const uint32_t vo = (uint32_t)(s * C::kTileBytes) >> 4;
              // k-step kk: P columns [8 kk, 8 kk + 8) (32 bytes of each row), V rows [kk kKStep, +kKStep)
#pragma unroll
              for (int kk = 0; kk < C::BN / C::kKStep; ++kk) {
                if constexpr (FP8)
                  mma_ts_f8(d_o, a_p + kk * 8, dv0 + vo + kk * ((C::kKStep * 128) >> 4), kIdO,
                            (j > 0 || kk > 0) ? 1u : 0u);
                else
                  mma_ts(d_o, a_p + kk * 8, dv0 + vo + kk * ((C::kKStep * 128) >> 4), kIdO,
                         (j > 0 || kk > 0) ? 1u : 0u);
              }
              // only the epilogue waits for O (the softmax learns of earlier PV products through
              // the S products issued after them), so only the last one is committed
              if (j == nb[t] - 1) mma_commit(&bars.o_done[t]);
              if (t == v_last) mma_commit(&bars.v_empty[s]);  // before the next S: V_j's slot refills sooner
            }
            __syncwarp();
          }
          if (jn < nb[t]) {
            if (elect_one()) issue_s(t, sn);
            __syncwarp();
          }
        }
        if (!ok) break;
        if (k_next) {
          if (elect_one()) mma_commit(&bars.k_empty[sn]);
          __syncwarp();
        }
      }
      if (elect_one()) mma_commit(&bars.teardown);
      __syncwarp();
      mbar_wait_drain(&bars.teardown, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // row within the tile = TMEM lane
    const int r0 = qblk * C::kRows + t * 128;
    const int row = r0 + r;
    const int nbt = nb[t];
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::col_s(t);
    const uint32_t t_o = tmem + lane_off + C::col_o(t);
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY;  // exponent reference, log2 units of scaled scores
    float l_sum = 0.f;        // sum of 2^(s * sl2 - m_ref) over the keys seen so far
    bool ok = true;
    for (int j = 0; j < nbt; ++j) {
      ok = mbar_wait(&bars.s_full[t], j & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {  // keep the warp converged for the .sync.aligned ops below
        ok = false;
        break;
      }
      tc_fence_after();
      // S_t, with the maximum of each 32 columns from the load itself
      uint32_t sr[4][32];
      float cmax[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_max(t_s + c * 32, sr[c], cmax[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c], cmax[c]);
      float mx = fmax3(fmax3(cmax[0], cmax[1], cmax[2]), cmax[3], -INFINITY);
      // Only blocks that reach past the tile's first row's last key (the
      // diagonal under the causal mask, one or two blocks) or past key sk - 1 need
      // masking: there a hidden score becomes -inf, so P = 0 (scale > 0), and the
      // row maximum is taken again over the scores that stay.
      const int kv0 = (jb + j) * C::BN;
      const bool need_mask = (CAUSAL && kv0 + C::BN - 1 > r0 + off) || kv0 + C::BN > sk;
      if (need_mask) {
        const int lim = (CAUSAL ? min(row + off, sk - 1) : sk - 1) - kv0;  // keep key column c iff c <= lim
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
        // Row maximum over eight independent chains of 16 scores (chain i takes
        // columns 2 i, 2 i + 1 of every 16-column group), then a tree: the
        // dependent chain is 8 + 2 instructions deep instead of 32.
        float mxc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          mxc[i] = fmaxf(__uint_as_float(sr[0][2 * i]), __uint_as_float(sr[0][2 * i + 1]));
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            mxc[i] = fmax3(mxc[i], __uint_as_float(sr[c >> 5][(c & 31) + 2 * i]),
                           __uint_as_float(sr[c >> 5][(c & 31) + 2 * i + 1]));
        mx = fmax3(fmax3(mxc[0], mxc[1], mxc[2]), fmax3(mxc[3], mxc[4], mxc[5]), fmaxf(mxc[6], mxc[7]));
      }
      float alpha = 1.f;
      bool move;
      if constexpr (FP8) {
        // integer reference, moved to ceil(max) once the max passes it by more than kP8Lag
        const float xm = mx * sl2;
        move = xm > m_ref + kP8Lag;
        if (move) {
          const float m_new = ceilf(xm);
          alpha = exp2_int_nonpos(m_ref - m_new);  // exact, so earlier rounded P stay exact multiples
          m_ref = m_new;
        }
      } else {
        const float m_new = fmaxf(m_ref, mx * sl2);
        move = m_new > m_ref + kRescaleThreshold;
        if (move) {
          alpha = ex2(m_ref - m_new);
          m_ref = m_new;
        }
      }
      const bool rescale = __any_sync(0xffffffffu, move && j > 0);
      // four partial row sums, so that the additions do not form one long chain
      float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // a row that has seen no key yet (possible within a key range) keeps m_ref = -inf and P = 0
      const float m_use = (m_ref == -INFINITY ? 0.f : m_ref) - (FP8 ? kP8Bias : 0.f);
      const float2 scale2 = make_float2(sl2, sl2), shift2 = make_float2(-m_use, -m_use);
      if constexpr (FP8) {
        // P as E4M3, four per column, over the first 32 columns of S_t; the row sum
        // takes P before rounding (the sum of the exponentials, as in the 16-bit path)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const int ch = 2 * half + (c >> 5), cc = c & 31;
            const float2 x0 =
                ffma2(make_float2(__uint_as_float(sr[ch][cc]), __uint_as_float(sr[ch][cc + 1])), scale2, shift2);
            const float2 x1 =
                ffma2(make_float2(__uint_as_float(sr[ch][cc + 2]), __uint_as_float(sr[ch][cc + 3])), scale2, shift2);
            const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y)), p1 = make_float2(ex2(x1.x), ex2(x1.y));
            sum4[(c >> 2) & 3] = fadd2(sum4[(c >> 2) & 3], fadd2(p0, p1));
            pk[c >> 2] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
          }
          tmem_st16(t_s + 16 * half, pk);
        }
      } else {
        // P as bf16 pairs over the first 64 columns of S_t (all of S_t is already in
        // registers), 32 scores at a time.
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 x =
                ffma2(make_float2(__uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1])), scale2, shift2);
            const float2 p = make_float2(ex2(x.x), ex2(x.y));
            sum4[(c >> 1) & 3] = fadd2(sum4[(c >> 1) & 3], p);
            pk[c >> 1] = pack_bf16x2(p.x, p.y);
          }
          if constexpr (DROP) {
            // keys kv0 + 32 ch + [0, 32) are 8 groups of 4: this lane draws groups qa and qa + 4 for
            // the quad's 4 rows, and the quad exchange leaves it its own row's bytes of all 8
            const uint32_t j4 = (uint32_t)(kv0 + 32 * ch) >> 2, i4 = (uint32_t)row >> 2, qa = lane & 3;
            const uint32_t thr4 = (uint32_t)a.drop_p256 * 0x01010101u;
            uint32_t x0[4], x1[4];
            philox::philox4x32_10(j4 + qa, i4, (uint32_t)bh, a.drop_offset, a.drop_rk, x0);
            philox::philox4x32_10(j4 + qa + 4, i4, (uint32_t)bh, a.drop_offset, a.drop_rk, x1);
            philox::quad_transpose(x0);
            philox::quad_transpose(x1);
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {  // x0[s4]: keys 4 s4 .. + 3 of the chunk; x1[s4]: 16 + 4 s4 ..
              const uint32_t k0m = philox::keep_bytes(x0[s4], thr4), k1m = philox::keep_bytes(x1[s4], thr4);
              pk[2 * s4] &= philox::pair_mask_lo(k0m);
              pk[2 * s4 + 1] &= philox::pair_mask_hi(k0m);
              pk[8 + 2 * s4] &= philox::pair_mask_lo(k1m);
              pk[8 + 2 * s4 + 1] &= philox::pair_mask_hi(k1m);
            }
          }
          tmem_st16(t_s + 16 * ch, pk);
        }
      }
      const float2 sum = fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3]));
      l_sum = l_sum * alpha + (sum.x + sum.y);
      if (rescale) {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(t_o + c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[t]);
    }
    if (ok && nbt > 0) ok = mbar_wait(&bars.o_done[t], 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (a.n_split > 1) {
      // O / l and the logsumexp of this key range, fp32, for the merge kernel
      // (a row that saw no key of the range: lse = -inf, and the merge skips it)
      const size_t prow = ((size_t)blockIdx.z * a.BH + bh) * Nq + row;
      if (ok && nbt > 0) {
        tc_fence_after();
        const float inv_l = l_sum > 0.f ? a.o_scale / l_sum : 0.f;
        float4* orow = reinterpret_cast<float4*>(a.o_part + prow * D);
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c, o);
          tmem_ld_wait(o);
          if (row < Nq)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              orow[(c >> 2) + i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                               __uint_as_float(o[4 * i + 2]) * inv_l,
                                               __uint_as_float(o[4 * i + 3]) * inv_l);
        }
      }
      if (ok && row < Nq)
        a.lse_part[prow] = nbt > 0 && l_sum > 0.f && (!VARLEN || row < sq) ? (m_ref - (FP8 ? kP8Bias : 0.f) + log2f(l_sum)) * kLn2 : -INFINITY;
    } else if (nbt == 0) {
      // every row of this tile is padding (another tile of the CTA is not)
      if (VARLEN && ok) zero_rows<D>(a, bh, r0, min(128, Nq - r0), r, 128);
    } else {  // nbt is uniform over the warpgroup, so every thread reaches the named barrier  // nbt is uniform over the warpgroup, so every thread reaches the named barrier
      uint8_t* stage = smem + C::kOffQ + t * C::kQSlotBytes;  // Q_t is no longer read by any MMA
      if (ok) {
        tc_fence_after();
        const float inv_l = a.o_scale / l_sum;
        const bool pad = VARLEN && row >= sq;  // a padding row among valid ones: o = 0
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(t_o + c, o);
          tmem_ld_wait(o);
          const int pn = c >> 6;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = ((c & 63) >> 3) + q4;  // 16-byte chunk within the 128-byte row
            const uint32_t addr = smem_u32(stage + pn * C::kPanelBytes + r * 128 + ((chunk ^ (r & 7)) << 4));
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = pad ? 0.f : __uint_as_float(o[q4 * 8 + i]) * inv_l;
            st_shared_v4(addr, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                         pack_bf16x2(f[6], f[7]));
          }
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(1 + t, 128);
      if (r == 0 && !*abort_flag) {
        for (int pn = 0; pn < C::kOPanels; ++pn)
          tma_store_3d(&a.tm_o, stage + pn * C::kPanelBytes, pn * 64, qblk * C::kRows + t * 128, bh);
        bulk_commit();
        bulk_wait_read0();  // the staging tile has been read; the writes finish on their own
      }
      if (ok && row < Nq)
        a.lse[(size_t)bh * Nq + row] =
            !VARLEN || row < sq ? (m_ref - (FP8 ? kP8Bias : 0.f) + log2f(l_sum)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpMma) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && bars.abort) atomicOr(a.status, 1u);
}

// Merge of the key ranges' results, one warp per query row: with
// m = max_z lse_z and w_z = e^(lse_z - m), o = sum_z w_z o_z / sum_z w_z and
// lse = m + ln sum_z w_z (the running-maximum update of chapter 08 of
// "FlashAttention and GPU Memory", for logsumexps, over all ranges at once).
// A range the row sees no key of has lse_z = -inf and is skipped; a row with
// no finite lse_z at all is a padding row: o = 0, lse = -inf.
template <int D>
__global__ void __launch_bounds__(256) fa_fwd_merge_kernel(const __grid_constant__ FwdArgs a) {
  constexpr int V = D / 32;  // values of the row per lane
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)a.BH * a.Nq;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int z = 0; z < a.n_split; ++z) m = fmaxf(m, a.lse_part[z * rows + row]);
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  float tot = 0.f;
  for (int z = 0; z < a.n_split; ++z) {
    const float lz = a.lse_part[z * rows + row];
    if (lz == -INFINITY) continue;
    const float w = expf(lz - m);
    tot += w;
    const float* oz = a.o_part + (z * rows + row) * D + lane * V;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] += w * oz[i];
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint32_t packed[V / 2];
#pragma unroll
  for (int i = 0; i < V / 2; ++i) packed[i] = pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.o) + (row * D + lane * V) * 2);
#pragma unroll
  for (int i = 0; i < V / 2; ++i) dst[i] = packed[i];
  if (lane == 0) a.lse[row] = tot > 0.f ? m + logf(tot) : -INFINITY;
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  auto kern = a.seqlens_q || a.seqlens_k ? fa_fwd_kernel<D, CAUSAL, true> : fa_fwd_kernel<D, CAUSAL, false>;
  if (a.drop_p256 > 0) kern = fa_fwd_kernel<D, CAUSAL, false, false, true>;  // dropout: no lengths, no key ranges
  int smem = FwdCfg<D>::kSmemBytes, threads = FwdCfg<D>::kThreads, rows = FwdCfg<D>::kRows;
  if constexpr (D == 128) {
    if (a.fp8) {  // 8-bit inputs: no lengths, no key ranges
      kern = fa_fwd_kernel<D, CAUSAL, false, true>;
      smem = FwdCfg<D, true>::kSmemBytes;
      threads = FwdCfg<D, true>::kThreads;
      rows = FwdCfg<D, true>::kRows;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(a.BH * ((a.Nq + rows - 1) / rows)), 1u, (unsigned)a.n_split);
  kern<<<grid, threads, smem, stream>>>(a);
  if (a.n_split > 1) {
    const long long rows = (long long)a.BH * a.Nq;
    fa_fwd_merge_kernel<D><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& args, int num_sms, cudaStream_t stream) {
  if (fwd_persist_applies(args)) return launch_fwd_persist(args, num_sms, stream);
  FwdArgs a = args;
  // a CTA's fixed cost (loads before the first product, epilogue) is about two key blocks of work
  const int rows = fwd_rows_per_cta(a.d), slots = num_sms * fwd_ctas_per_sm(a.d);
  a.head_group = pick_head_group(a.BH, (a.Nq + rows - 1) / rows, a.causal != 0, slots, 2.0);
  if (a.d == 64) return a.causal ? launch_fwd_t<64, true>(a, stream) : launch_fwd_t<64, false>(a, stream);
  return a.causal ? launch_fwd_t<128, true>(a, stream) : launch_fwd_t<128, false>(a, stream);
}

}  // namespace fa
