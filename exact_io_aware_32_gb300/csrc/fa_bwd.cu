// Backward pass of exact attention on sm_103a.
//
// The pages keep only O and the per-row statistics from the forward pass and
// rebuild S and P block by block from Q, K and V ("FlashAttention and GPU
// Memory", chapter 09). With lse_i the row logsumexp, for a block of keys j
// and a block of queries i:
//   S^T = K_j Q_i^T,  P^T = exp(scale S^T - lse_i),  dP^T = V_j dO_i^T,
//   dS^T = P^T o (dP^T - D_i)   with D_i = dO_i . O_i,
//   dV_j += P^T dO_i,  dK_j += scale dS^T Q_i,  dQ_i += scale dS K_j.
// (The chain rule of softmax; D_i = sum_k P_ik dP_ik equals dO_i . O_i.)
//
// Three kernels run in order on one stream:
//   1. bwd_prep:    D_i = dO_i . O_i (fp32), and zero the fp32 dQ accumulator
//   2. bwd_main:    one CTA per 128-key block; loops over 128-row query blocks
//   3. bwd_dq_cast: dQ accumulator (fp32) -> dq (bf16)
//
// bwd_main warp roles (320 threads): warps 0-3 (warpgroup 0) turn S^T and dP^T
// into P^T (written back to tensor memory as bf16) and dS^T (written to shared
// memory as bf16); warps 4-7 (warpgroup 1) drain each dQ block from tensor
// memory into the fp32 accumulator with atomic adds; warp 8 issues TMA loads;
// warp 9 issues the tcgen05 MMAs. Thread r of a warpgroup owns TMEM lane r:
// key r of the block for S^T, dP^T, dK, dV; for the dQ block, feature r at
// d = 128 (the product is formed transposed, dQ^T = K^T dS^T, so that a warp's
// atomics hit one contiguous row) and query r at d = 64.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

using namespace fa::ptx;

constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct BwdCfg {
  static constexpr int BK = 128;  // keys per CTA
  static constexpr int BQ = 128;  // queries per iteration
  static constexpr int kPanelBytes = 128 * 128;
  static constexpr int kTileBytes = (D / 64) * kPanelBytes;  // 128 rows x D bf16
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;     // 2 stages
  static constexpr int kOffDO = kOffQ + 2 * kTileBytes;  // 2 stages
  static constexpr int kOffDS = kOffDO + 2 * kTileBytes;  // dS^T: 128 keys x 128 queries bf16, 2 panels
  static constexpr int kOffLse = kOffDS + 2 * kPanelBytes;  // 128 fp32 (log2 units)
  static constexpr int kOffDv = kOffLse + 512;              // 128 fp32
  static constexpr int kOffBar = kOffDv + 512;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  // TMEM columns
  static constexpr uint32_t kColS = 0;     // S^T fp32, 128 cols; P^T bf16 in its first 64
  static constexpr uint32_t kColDP = 128;  // dP^T fp32, 128 cols
  static constexpr uint32_t kColDV = 256;  // dV accumulator, D cols
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr uint32_t kColDQ = D == 128 ? kColDP : 256 + 2 * D;  // dQ block (fp32, D cols)
};

struct BwdBarriers {
  uint64_t kv_full;
  uint64_t qd_full[2], qd_empty[2];
  uint64_t s_full, dp_full, ds_ready, dq_full, mma_done, dq_free;
  uint64_t teardown;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void red_add_f32(float* p, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Writes one 128-byte-swizzled row of bf16 pairs: 'words' 32-bit words
// (2 bf16 each) starting at 16-byte chunk 'chunk0' of row r of a panel.
__device__ __forceinline__ void st_swizzled_row(uint8_t* panel, int r, int chunk0, const uint32_t* w, int nchunks) {
#pragma unroll
  for (int c = 0; c < nchunks; ++c) {
    const int chunk = chunk0 + c;
    st_shared_v4(smem_u32(panel + r * 128 + (((chunk & 7) ^ (r & 7)) << 4)), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                 w[4 * c + 3]);
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(320, 1) fa_bwd_main_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBarriers& bars = *reinterpret_cast<BwdBarriers*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars.abort;
  float* s_lse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* s_dv = reinterpret_cast<float*>(smem + C::kOffDv);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int bh = blockIdx.x;
  const int kblk = blockIdx.y;  // heaviest key blocks (most query blocks under the causal mask) first
  const int nq = (N + C::BQ - 1) / C::BQ;
  const int i_start = CAUSAL ? kblk : 0;  // BQ == BK: query block i sees key block j iff i >= j
  const int n_iter = nq - i_start;

  if (threadIdx.x == 0) {
    bars.abort = 0;
    mbar_init(&bars.kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.qd_full[s], 1);
      mbar_init(&bars.qd_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.ds_ready, 128);
    mbar_init(&bars.dq_full, 1);
    mbar_init(&bars.mma_done, 1);
    mbar_init(&bars.dq_free, 128);
    mbar_init(&bars.teardown, 1);
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

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_q);
      tma_prefetch_desc(&a.tm_do);
      mbar_arrive_expect_tx(&bars.kv_full, 2 * C::kTileBytes);
      for (int pn = 0; pn < D / 64; ++pn) {
        tma_load_3d(smem + C::kOffK + pn * C::kPanelBytes, &a.tm_k, &bars.kv_full, pn * 64, kblk * C::BK, bh);
        tma_load_3d(smem + C::kOffV + pn * C::kPanelBytes, &a.tm_v, &bars.kv_full, pn * 64, kblk * C::BK, bh);
      }
      int issued = 0;
      for (int it = 0; it < n_iter; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&bars.qd_empty[s], ph ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&bars.qd_full[s], 2 * C::kTileBytes);
        const int q0 = (i_start + it) * C::BQ;
        for (int pn = 0; pn < D / 64; ++pn) {
          tma_load_3d(smem + C::kOffQ + s * C::kTileBytes + pn * C::kPanelBytes, &a.tm_q, &bars.qd_full[s],
                      pn * 64, q0, bh);
          tma_load_3d(smem + C::kOffDO + s * C::kTileBytes + pn * C::kPanelBytes, &a.tm_do, &bars.qd_full[s],
                      pn * 64, q0, bh);
        }
        issued = it + 1;
      }
      mbar_wait_drain(&bars.kv_full, 0);
      for (int i = max(0, issued - 2); i < issued; ++i) mbar_wait_drain(&bars.qd_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdKK = idesc_bf16(128, 128, false, false);  // S^T, dP^T: both operands K-major
      constexpr uint32_t kIdTS = idesc_bf16(128, D, false, true);     // dV: P^T from TMEM, dO MN-major
      constexpr uint32_t kIdKM = idesc_bf16(128, D, false, true);     // dK: dS^T K-major, Q MN-major
      constexpr uint32_t kIdMM = idesc_bf16(128, D, true, true);      // dQ (or dQ^T): both operands MN-major
      const uint32_t k_base = smem_u32(smem + C::kOffK), v_base = smem_u32(smem + C::kOffV);
      const uint32_t q_base = smem_u32(smem + C::kOffQ), do_base = smem_u32(smem + C::kOffDO);
      const uint32_t ds_base = smem_u32(smem + C::kOffDS);
      bool ok = mbar_wait(&bars.kv_full, 0, abort_flag);
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        const uint32_t qs = q_base + s * C::kTileBytes, dos = do_base + s * C::kTileBytes;
        if (!(ok = mbar_wait(&bars.qd_full[s], ph, abort_flag))) break;
        // S^T and P^T share columns; dS^T in shared memory is rewritten: the previous
        // block's dV, dK and dQ products must be complete.
        if (it > 0 && !(ok = mbar_wait(&bars.mma_done, (it - 1) & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kPanelBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColS, sdesc_sw128(k_base + off, 16, 1024), sdesc_sw128(qs + off, 16, 1024), kIdKK,
                 kk > 0);
        }
        mma_commit(&bars.s_full);
        // dP^T shares columns with the previous dQ block when D == 128.
        if (D == 128 && it > 0 && !(ok = mbar_wait(&bars.dq_free, (it - 1) & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kPanelBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColDP, sdesc_sw128(v_base + off, 16, 1024), sdesc_sw128(dos + off, 16, 1024), kIdKK,
                 kk > 0);
        }
        mma_commit(&bars.dp_full);
        if (!(ok = mbar_wait(&bars.ds_ready, it & 1, abort_flag))) break;
        tc_fence_after();
        if (D == 64 && it > 0 && !(ok = mbar_wait(&bars.dq_free, (it - 1) & 1, abort_flag))) break;
        tc_fence_after();
        // dQ first, so that its drain overlaps dV and dK. K = 128 keys.
        // d = 128: dQ^T = K^T dS^T (lane = feature), so the drain's atomics are
        //          contiguous along d; d = 64: dQ = dS K (lane = query).
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint64_t dsd = sdesc_sw128(ds_base + kk * 2048, C::kPanelBytes, 1024);
          const uint64_t kd = sdesc_sw128(k_base + kk * 2048, C::kPanelBytes, 1024);
          if (D == 128)
            mma_ss(tmem + C::kColDQ, kd, dsd, kIdMM, kk > 0);
          else
            mma_ss(tmem + C::kColDQ, dsd, kd, kIdMM, kk > 0);
        }
        mma_commit(&bars.dq_full);
        // dV += P^T dO_i   (K = 128 queries, 16 per instruction)
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          mma_ts(tmem + C::kColDV, tmem + C::kColS + kk * 8, sdesc_sw128(dos + kk * 2048, C::kPanelBytes, 1024),
                 kIdTS, (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q_i
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kPanelBytes + (kk & 3) * 32;
          mma_ss(tmem + C::kColDK, sdesc_sw128(ds_base + off, 16, 1024),
                 sdesc_sw128(qs + kk * 2048, C::kPanelBytes, 1024), kIdKM, (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars.mma_done);
        mma_commit(&bars.qd_empty[s]);
      }
      mma_commit(&bars.teardown);
      mbar_wait_drain(&bars.teardown, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ warpgroup 0: P^T, dS^T, then dV out
    const int r = threadIdx.x;  // key within the block
    const int key = kblk * C::BK + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kColS, t_dp = tmem + lane_off + C::kColDP;
    const float sl2 = a.scale_log2;
    uint8_t* ds_panel0 = smem + C::kOffDS;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int q0 = (i_start + it) * C::BQ;
      {
        const int q = q0 + r;
        const size_t gi = (size_t)bh * N + q;
        const float l2 = q < N ? a.lse[gi] * kLog2e : INFINITY;  // exp2(x - inf) = 0 masks rows past N
        const float dsum = q < N ? a.Dsum[gi] : 0.f;
        if (it > 0) named_bar_sync(1, 128);  // every thread has finished reading the previous block's values
        s_lse[r] = l2;
        s_dv[r] = dsum;
      }
      named_bar_sync(1, 128);
      ok = mbar_wait(&bars.s_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T row r as bf16 pairs; the same rounded values feed dV (through TMEM) and dS.
      uint32_t pk[64];
      {
        const bool diag = CAUSAL && (q0 == kblk * C::BK);
        const bool key_ok = key < N;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t sr[32];
          tmem_ld32(t_s + c0, sr);
          tmem_ld_wait(sr);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float v0 = ex2(fmaf(__uint_as_float(sr[c]), sl2, -s_lse[c0 + c]));
            float v1 = ex2(fmaf(__uint_as_float(sr[c + 1]), sl2, -s_lse[c0 + c + 1]));
            // causal: query q0 + c is visible to key q0 + r only if c >= r
            if ((diag && c0 + c < r) || !key_ok) v0 = 0.f;
            if ((diag && c0 + c + 1 < r) || !key_ok) v1 = 0.f;
            pk[(c0 + c) >> 1] = pack_bf16x2(v0, v1);
          }
        }
        // All of S^T has been read: P^T may overwrite its first 64 columns.
        tmem_st32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      }
      ok = mbar_wait(&bars.dp_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t dp[32];
        tmem_ld32(t_dp + c0, dp);
        tmem_ld_wait(dp);
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const uint32_t pp = pk[(c0 + c) >> 1];
          const float d0 = __uint_as_float(pp << 16) * (__uint_as_float(dp[c]) - s_dv[c0 + c]);
          const float d1 = __uint_as_float(pp & 0xFFFF0000u) * (__uint_as_float(dp[c + 1]) - s_dv[c0 + c + 1]);
          w[c >> 1] = pack_bf16x2(d0, d1);
        }
        // dS^T row r, queries c0..c0+31: panel c0 / 64, chunks (c0 % 64) / 8 .. + 3
        st_swizzled_row(ds_panel0 + (c0 >> 6) * C::kPanelBytes, r, (c0 & 63) >> 3, w, 4);
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.ds_ready);
    }
    // dV epilogue: wait for the last products, then dV (fp32, TMEM) -> bf16 -> TMA store.
    if (ok && n_iter > 0) ok = mbar_wait(&bars.mma_done, (n_iter - 1) & 1, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    uint8_t* stage = smem + C::kOffQ;  // free once every product has completed
    if (ok && n_iter > 0) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + C::kColDV + c, o);
        tmem_ld_wait(o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
        st_swizzled_row(stage + (c >> 6) * C::kPanelBytes, r, (c & 63) >> 3, w, 4);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (r == 0 && n_iter > 0 && !*abort_flag) {
      for (int pn = 0; pn < D / 64; ++pn)
        tma_store_3d(&a.tm_dv, stage + pn * C::kPanelBytes, pn * 64, kblk * C::BK, bh);
      bulk_commit();
      bulk_wait0();
    }
  } else {
    // ------------------------------------------------------------ warpgroup 1: dQ drain, then dK out
    const int r = threadIdx.x - 128;  // query within the block (dQ) / key within the block (dK)
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float scale = a.scale;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      ok = mbar_wait(&bars.dq_full, it & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int q0 = (i_start + it) * C::BQ;
      if (D == 128) {
        // lane r = feature r; columns = the block's 128 queries. Each warp adds
        // 32 consecutive floats of one dQ row per instruction.
        float* col = a.dqacc + ((size_t)bh * N + q0) * D + r;
#pragma unroll 1
        for (int c0 = 0; c0 < C::BQ; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + C::kColDQ + c0, o);
          tmem_ld_wait(o);
          const int nvalid = min(32, N - (q0 + c0));
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nvalid) red_add_f32(col + (size_t)(c0 + i) * D, __uint_as_float(o[i]) * scale);
        }
      } else {
        const int q = q0 + r;  // lane r = query r
        float* dst = a.dqacc + ((size_t)bh * N + q) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + C::kColDQ + c, o);
          tmem_ld_wait(o);
          if (q < N) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              red_add_v4(dst + c + i, __uint_as_float(o[i]) * scale, __uint_as_float(o[i + 1]) * scale,
                         __uint_as_float(o[i + 2]) * scale, __uint_as_float(o[i + 3]) * scale);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars.dq_free);
    }
    if (ok && n_iter > 0) ok = mbar_wait(&bars.mma_done, (n_iter - 1) & 1, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    // dK epilogue, once the last products have completed
    uint8_t* stage = smem + C::kOffDO;
    if (ok && n_iter > 0) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + C::kColDK + c, o);
        tmem_ld_wait(o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * scale, __uint_as_float(o[2 * i + 1]) * scale);
        st_swizzled_row(stage + (c >> 6) * C::kPanelBytes, r, (c & 63) >> 3, w, 4);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(2, 128);
    if (r == 0 && n_iter > 0 && !*abort_flag) {
      for (int pn = 0; pn < D / 64; ++pn)
        tma_store_3d(&a.tm_dk, stage + pn * C::kPanelBytes, pn * 64, kblk * C::BK, bh);
      bulk_commit();
      bulk_wait0();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && bars.abort) atomicOr(a.status, 2u);
}

// D_i = dO_i . O_i in fp32, and zero the fp32 dQ accumulator. Each thread
// handles 8 consecutive elements of one row; D / 8 threads share a row.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int kThreadsPerRow = D / 8;
  const long long rows = (long long)a.BH * a.N;
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
    float4* z = reinterpret_cast<float4*>(a.dqacc + row * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kThreadsPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) a.Dsum[row] = acc;
}

// dq (bf16) = dQ accumulator (fp32, already scaled). 8 elements per thread.
__global__ void __launch_bounds__(256) fa_bwd_dq_cast_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                             long long n8) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= n8) return;
  const float4 x = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 y = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 w;
  w.x = pack_bf16x2(x.x, x.y);
  w.y = pack_bf16x2(x.z, x.w);
  w.z = pack_bf16x2(y.x, y.y);
  w.w = pack_bf16x2(y.z, y.w);
  reinterpret_cast<uint4*>(dq)[i] = w;
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const long long rows = (long long)a.BH * a.N;
  const int rows_per_block = 256 / (D / 8);
  fa_bwd_prep_kernel<D><<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = fa_bwd_main_kernel<D, CAUSAL>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<dim3((unsigned)a.BH, (unsigned)((a.N + C::BK - 1) / C::BK)), 320, C::kSmemBytes, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n8 = rows * D / 8;
  fa_bwd_dq_cast_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, stream>>>(a.dqacc, static_cast<uint16_t*>(a.dq), n8);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, int /*num_sms*/, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_bwd_t<64, true>(a, stream) : launch_bwd_t<64, false>(a, stream);
  return a.causal ? launch_bwd_t<128, true>(a, stream) : launch_bwd_t<128, false>(a, stream);
}

}  // namespace fa
