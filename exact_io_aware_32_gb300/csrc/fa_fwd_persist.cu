// Persistent forward pass for d = 64 on sm_103a.
//
// The same computation as fa_fwd.cu's kernel (the blocked loop of "FlashAttention
// and GPU Memory", chapter 07, with the running-maximum softmax of chapter 08):
// per 128-row query tile and 128-key block, S = Q K^T on tcgen05 into TMEM, the
// softmax with one TMEM lane (= one query row) per thread, O += P V with P read
// back from TMEM as bf16, and at the end O / l and the row logsumexp.
//
// At d = 64 a tile's products take half the time of d = 128 while its fixed
// costs do not shrink: loading Q and the first K before the first product,
// and reading O out of TMEM and storing it after the last. With one CTA per tile,
// short rows (N = 1024 under the causal mask: 4.5 key blocks a tile on
// average) spent about a quarter of each CTA's life in those two phases. Here
// each CTA (two per SM) runs a sequence of tiles instead, so that they overlap
// the neighbouring tiles' work:
//   - Q has two slots: the next tile's Q is loaded while the current tile runs;
//   - P has TMEM columns of its own, apart from S: once the softmax has read S
//     of a block into registers, S of the next block (of this tile or the next)
//     is computed while the softmax works, so the softmax warps never wait for
//     two products in a row;
//   - the K/V rings, their barriers and the S/P barriers count key blocks over
//     the CTA's whole run, so the pipeline never drains between tiles.
// Tiles are dealt to CTAs statically, in rounds of one tile per CTA, every
// other round in reverse CTA order: under the causal mask the tiles are ordered
// heaviest first within each head group, so a CTA that takes a heavy tile in one
// round takes a light one in the next.
//
// Warp roles (192 threads): warps 0-3 softmax and epilogue, warp 4 TMA loads,
// warp 5 MMAs and the TMEM allocation. Used for the plain d = 64 forward (no
// padding masks, no key ranges, no dropout); the other forms keep fa_fwd.cu's kernel.
#include <algorithm>

#include "fa_internal.h"
#include "block_order.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace fa::ptx;

constexpr float kLn2 = 0.693147180559945309417f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units, as in fa_fwd.cu

struct PCfg {
  static constexpr int D = 64;
  static constexpr int BN = 128;                    // keys per block
  static constexpr int kTileBytes = 128 * 128;      // 128 rows x 64 bf16: one 128-byte-swizzled panel
  static constexpr int kKStages = 2, kVStages = 3;  // V is read last, so it gets the deeper ring
  static constexpr int kOffQ = 0;                   // two Q slots (each also stages its tile's O)
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  // No alignment slack (two CTAs must share an SM's 228 KB): the kernel checks
  // that dynamic shared memory starts on a 1024-byte boundary.
  static constexpr int kSmemBytes = kOffBar + 256;
  static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs must fit an SM's shared memory");
  static constexpr uint32_t kColS = 0;    // S fp32, 128 columns
  static constexpr uint32_t kColP = 128;  // P as bf16 pairs, 64 columns
  static constexpr uint32_t kColO = 192;  // O fp32, 64 columns
  static constexpr uint32_t kTmemCols = 256;
  static constexpr int kThreads = 192;
  static constexpr int kWarpTma = 4, kWarpMma = 5;
};

struct PBars {
  uint64_t q_full[2], q_free[2];
  uint64_t k_full[2], k_empty[2], v_full[3], v_empty[3];
  uint64_t s_full, s_free, p_full, pv_done, o_free;
  uint64_t teardown;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PBars) <= 256, "barriers exceed their shared memory");

struct PTile {
  int bh, qblk, nb;  // head, query block, key blocks it sees
};

// The i-th tile of this CTA (nb = 0 past the end of its sequence).
template <bool CAUSAL>
__device__ __forceinline__ PTile ptile(const FwdArgs& a, int i, int nqblk) {
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const long long L = (long long)i * G + ((i & 1) ? G - 1 - c : c);
  PTile t{0, 0, 0};
  if (L >= (long long)a.BH * nqblk) return t;
  int blk;
  grouped_index((int)L, a.BH, nqblk, a.head_group, t.bh, blk);
  t.qblk = CAUSAL ? nqblk - 1 - blk : blk;
  const int off = a.Nk - a.Nq;  // causal: query row i sees keys 0 .. i + off
  const int r0 = t.qblk * 128;
  const int last_key = CAUSAL ? min(min(r0 + 127, a.Nq - 1) + off, a.Nk - 1) : a.Nk - 1;
  t.nb = last_key / PCfg::BN + 1;
  return t;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(PCfg::kThreads, 2) fa_fwd_persist_kernel(const __grid_constant__ FwdArgs a) {
  using C = PCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const int nqblk = (a.Nq + 127) / 128;
  if (ptile<CAUSAL>(a, 0, nqblk).nb == 0) return;  // no tile for this CTA (uniform)
  if (smem_u32(smem) & 1023u) {  // uniform over the CTA: every thread leaves before any barrier
    if (threadIdx.x == 0) atomicOr(a.status, 16u);
    return;
  }
  PBars& bars = *reinterpret_cast<PBars*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    bars.abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_free[s], 1);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, 128);
    mbar_init(&bars.p_full, 128);
    mbar_init(&bars.pv_done, 1);
    mbar_init(&bars.o_free, 128);
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
    // Per tile: Q into its slot (once the tile two back has stored its O from
    // there), then K and V of each key block into the rings.
    if (elect_one()) {
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
    }
    __syncwarp();
    int g = 0, nk = 0, nv = 0, q_last[2] = {-1, -1};  // K, V loads issued; the last tile per Q slot
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const PTile t = ptile<CAUSAL>(a, i, nqblk);
      if (t.nb == 0) break;
      const int slot = i & 1;
      if (!(ok = warp_wait(&bars.q_free[slot], ((i >> 1) & 1) ^ 1, abort_flag))) break;
      // test hook: without the first Q tile, the MMA warp's first wait expires
      if (i > 0 || a.test_fault != 1) {
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.q_full[slot], C::kTileBytes);
          tma_load_3d(smem + C::kOffQ + slot * C::kTileBytes, &a.tm_q, &bars.q_full[slot], 0, t.qblk * 128, t.bh);
        }
        __syncwarp();
        q_last[slot] = i;
      }
      for (int j = 0; j < t.nb; ++j, ++g) {
        const int ks = g % C::kKStages, vs = g % C::kVStages;
        if (!(ok = warp_wait(&bars.k_empty[ks], ((g / C::kKStages) & 1) ^ 1, abort_flag))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.k_full[ks], C::kTileBytes);
          tma_load_3d(smem + C::kOffK + ks * C::kTileBytes, &a.tm_k, &bars.k_full[ks], 0, j * C::BN, t.bh);
        }
        __syncwarp();
        nk = g + 1;
        if (!(ok = warp_wait(&bars.v_empty[vs], ((g / C::kVStages) & 1) ^ 1, abort_flag))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.v_full[vs], C::kTileBytes);
          tma_load_3d(smem + C::kOffV + vs * C::kTileBytes, &a.tm_v, &bars.v_full[vs], 0, j * C::BN, t.bh);
        }
        __syncwarp();
        nv = g + 1;
      }
    }
    // Let every issued copy land before the CTA can exit: the last Q of each slot
    // and the last loads of each ring (an earlier load's slot was refilled only
    // after its reader completed, so it has landed).
    for (int s = 0; s < 2; ++s)
      if (q_last[s] >= 0) mbar_wait_drain(&bars.q_full[s], (q_last[s] >> 1) & 1);
    for (int x = max(0, nk - C::kKStages); x < nk; ++x)
      mbar_wait_drain(&bars.k_full[x % C::kKStages], (x / C::kKStages) & 1);
    for (int x = max(0, nv - C::kVStages); x < nv; ++x)
      mbar_wait_drain(&bars.v_full[x % C::kVStages], (x / C::kVStages) & 1);
  } else if (warp == C::kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // Per key block g: S of block g + 1 as soon as the softmax has read S of
    // block g (and, for a tile's first block, its Q has landed), then O += P V
    // once P of block g is written. At a tile's last block P V goes first, so
    // that the epilogue can read O out sooner, and S of the next tile's first
    // block follows.
    constexpr uint32_t kIdS = idesc_bf16(128, C::BN, false, false);  // Q, K both K-major
    constexpr uint32_t kIdO = idesc_bf16(128, C::D, false, true);    // P from TMEM, V MN-major
    const uint64_t dq0 = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dk0 = sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dv0 = sdesc_sw128(smem_u32(smem + C::kOffV), C::kTileBytes, 1024);
    auto issue_s = [&](int slot, int g) {  // by the elected lane
      const uint32_t qo = (uint32_t)(slot * C::kTileBytes) >> 4;
      const uint32_t ko = (uint32_t)((g % C::kKStages) * C::kTileBytes) >> 4;
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk)  // each k-step reads 32 bytes of every row
        mma_ss(tmem + C::kColS, dq0 + qo + kk * 2, dk0 + ko + kk * 2, kIdS, kk > 0);
      mma_commit(&bars.s_full);
      mma_commit(&bars.k_empty[g % C::kKStages]);  // S is K's only reader
    };
    // S of block g + 1 (Q slot 'slot'); 'new_tile' adds the wait for that tile's Q
    auto next_s = [&](int g, int slot, bool new_tile, int i_next) -> bool {
      const int ks = (g + 1) % C::kKStages;
      bool w = warp_wait2(&bars.s_free, g & 1, &bars.k_full[ks], ((g + 1) / C::kKStages) & 1, abort_flag);
      if (w && new_tile) w = warp_wait(&bars.q_full[slot], (i_next >> 1) & 1, abort_flag);
      if (!w) return false;
      tc_fence_after();
      if (elect_one()) issue_s(slot, g + 1);
      __syncwarp();
      return true;
    };
    bool ok = warp_wait2(&bars.q_full[0], 0, &bars.k_full[0], 0, abort_flag);
    if (ok) {
      tc_fence_after();
      if (elect_one()) issue_s(0, 0);
      __syncwarp();
    }
    const uint32_t d_o = tmem + C::kColO;
    int g = 0;
    PTile t = ptile<CAUSAL>(a, 0, nqblk);
    for (int i = 0; ok && t.nb > 0; ++i) {
      const int slot = i & 1;
      const PTile tn = ptile<CAUSAL>(a, i + 1, nqblk);
      for (int j = 0; j < t.nb; ++j, ++g) {
        const bool last = j + 1 == t.nb;
        if (!last && !(ok = next_s(g, slot, false, 0))) break;
        const int vs = g % C::kVStages;
        ok = warp_wait2(&bars.p_full, g & 1, &bars.v_full[vs], (g / C::kVStages) & 1, abort_flag);
        // the first P V of a tile overwrites O: the previous tile's epilogue has read it out
        if (ok && j == 0 && i > 0) ok = warp_wait(&bars.o_free, (i - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t vo = (uint32_t)(vs * C::kTileBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)  // P columns [8 kk, 8 kk + 8), V rows [16 kk, 16 kk + 16)
            mma_ts(d_o, tmem + C::kColP + kk * 8, dv0 + vo + kk * ((16 * 128) >> 4), kIdO,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars.pv_done);
          mma_commit(&bars.v_empty[vs]);
        }
        __syncwarp();
        if (last && tn.nb > 0 && !(ok = next_s(g, slot ^ 1, true, i + 1))) break;
      }
      t = tn;
    }
    if (elect_one()) mma_commit(&bars.teardown);
    __syncwarp();
    mbar_wait_drain(&bars.teardown, 0);
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = warp * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS;
    const uint32_t t_p = tmem + lane_off + C::kColP;
    const uint32_t t_o = tmem + lane_off + C::kColO;
    const float sl2 = a.scale_log2;
    const int off = a.Nk - a.Nq;
    bool ok = true;
    int g = 0;
    for (int i = 0;; ++i) {
      const PTile t = ptile<CAUSAL>(a, i, nqblk);
      if (t.nb == 0) break;
      const int slot = i & 1;
      const int r0 = t.qblk * 128, row = r0 + r;
      float m_ref = -INFINITY;  // exponent reference, log2 units of scaled scores
      float l_sum = 0.f;        // sum of 2^(s * sl2 - m_ref) over the keys seen so far
      for (int j = 0; j < t.nb; ++j, ++g) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full, g & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        // S, with the maximum of each 32 columns from the load itself
        uint32_t sr[4][32];
        float cmax[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_max(t_s + c * 32, sr[c], cmax[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c], cmax[c]);
        tc_fence_before();
        mbar_arrive(&bars.s_free);  // S is in registers: the next block's S may overwrite it
        float mx = fmax3(fmax3(cmax[0], cmax[1], cmax[2]), cmax[3], -INFINITY);
        // only blocks that reach past the tile's first row's last key, or past
        // the last key, need masking: a hidden score becomes -inf, so P = 0, and
        // the row maximum is taken again over the scores that stay
        const int kv0 = j * C::BN;
        if ((CAUSAL && kv0 + C::BN - 1 > r0 + off) || kv0 + C::BN > a.Nk) {
          const int lim = (CAUSAL ? min(row + off, a.Nk - 1) : a.Nk - 1) - kv0;  // keep column c iff c <= lim
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
          // row maximum over eight chains of 16 scores, then a tree
          float mxc[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            mxc[q] = fmaxf(__uint_as_float(sr[0][2 * q]), __uint_as_float(sr[0][2 * q + 1]));
#pragma unroll
          for (int c = 16; c < 128; c += 16)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              mxc[q] = fmax3(mxc[q], __uint_as_float(sr[c >> 5][(c & 31) + 2 * q]),
                             __uint_as_float(sr[c >> 5][(c & 31) + 2 * q + 1]));
          mx = fmax3(fmax3(mxc[0], mxc[1], mxc[2]), fmax3(mxc[3], mxc[4], mxc[5]), fmaxf(mxc[6], mxc[7]));
        }
        float alpha = 1.f;
        const float m_new = fmaxf(m_ref, mx * sl2);
        const bool move = m_new > m_ref + kRescaleThreshold;
        if (move) {
          alpha = ex2(m_ref - m_new);
          m_ref = m_new;
        }
        const bool rescale = __any_sync(0xffffffffu, move && j > 0);
        float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
        const float2 scale2 = make_float2(sl2, sl2), shift2 = make_float2(-m_ref, -m_ref);
        // P as bf16 pairs, 32 scores at a time. P and O of the previous block are free
        // once its P V has completed (a tile's first block: the previous tile's
        // epilogue waited for that already); the first two chunks are computed before
        // that wait, packed in place (pair c / 2 of a chunk into word c / 2, already read).
        auto chunk = [&](int ch) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 x =
                ffma2(make_float2(__uint_as_float(sr[ch][c]), __uint_as_float(sr[ch][c + 1])), scale2, shift2);
            const float2 p = make_float2(ex2(x.x), ex2(x.y));
            sum4[(c >> 1) & 3] = fadd2(sum4[(c >> 1) & 3], p);
            sr[ch][c >> 1] = pack_bf16x2(p.x, p.y);
          }
        };
        auto store = [&](int ch) {
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) pk[q] = sr[ch][q];
          tmem_st16(t_p + 16 * ch, pk);
        };
        chunk(0);
        chunk(1);
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars.pv_done, (g - 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
        }
        store(0);
        store(1);
        chunk(2);
        store(2);
        chunk(3);
        store(3);
        const float2 sum = fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3]));
        l_sum = l_sum * alpha + (sum.x + sum.y);
        if (rescale) {
#pragma unroll 1
          for (int c = 0; c < C::D; c += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + c, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(t_o + c, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.p_full);
      }
      // Epilogue of tile i; every thread of the warpgroup runs it (named barriers).
      if (ok) ok = mbar_wait(&bars.pv_done, (g - 1) & 1, abort_flag);  // the tile's last P V
      ok = __all_sync(0xffffffffu, ok);
      uint8_t* stage = smem + C::kOffQ + slot * C::kTileBytes;  // this tile's Q: its last S has completed
      if (ok) {
        tc_fence_after();
        uint32_t o[2][32];
        tmem_ld32(t_o, o[0]);
        tmem_ld32(t_o + 32, o[1]);
        tmem_ld_wait(o[0]);
        tmem_ld_wait(o[1]);
        tc_fence_before();
        mbar_arrive(&bars.o_free);  // O is in registers: tile i + 1 may accumulate there
        const float inv_l = 1.f / l_sum;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = 4 * h + q4;  // 16-byte chunk within the 128-byte row
            const uint32_t addr = smem_u32(stage + r * 128 + ((chunk ^ (r & 7)) << 4));
            float f[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(o[h][q4 * 8 + q]) * inv_l;
            st_shared_v4(addr, pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                         pack_bf16x2(f[6], f[7]));
          }
        fence_proxy_async_smem();
      }
      named_bar_sync(1, 128);
      if (r == 0) {
        if (!*abort_flag) {
          tma_store_3d(&a.tm_o, stage, 0, r0, t.bh);
          bulk_commit();
          bulk_wait_read0();  // the staging tile has been read; the writes finish on their own
        }
        mbar_arrive(&bars.q_free[slot]);  // the slot may take the Q of tile i + 2
      }
      if (ok && row < a.Nq) a.lse[(size_t)t.bh * a.Nq + row] = (m_ref + log2f(l_sum)) * kLn2;
      if (!named_bar_and(1, 128, ok)) break;  // the four warps agree whether to go on
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpMma) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && bars.abort) atomicOr(a.status, 1u);
}

}  // namespace

bool fwd_persist_applies(const FwdArgs& a) {
  return a.d == 64 && !a.fp8 && a.drop_p256 == 0 && !a.seqlens_q && !a.seqlens_k && a.n_split <= 1;
}

cudaError_t launch_fwd_persist(const FwdArgs& args, int num_sms, cudaStream_t stream) {
  FwdArgs a = args;
  const int nqblk = (a.Nq + 127) / 128;
  const long long tiles = (long long)a.BH * nqblk;
  const int ctas = (int)std::min<long long>(tiles, 2ll * num_sms);
  // About one round of tiles per head group, so that the CTAs of a round share K
  // and V in L2. When the K and V of every head fit in L2 together (64 MB here,
  // half of it), one group instead: the heaviest tiles of all heads go first, and
  // with few rounds the rounds balance better (the last one is the lightest).
  const double kv_bytes = 2.0 * 2.0 * (double)a.BH * (double)a.Nk * (double)a.d;
  a.head_group = kv_bytes <= 64.0e6 ? a.BH : std::max(1, std::min(a.BH, ctas / nqblk));
  auto kern = a.causal ? fa_fwd_persist_kernel<true> : fa_fwd_persist_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)ctas, PCfg::kThreads, PCfg::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
