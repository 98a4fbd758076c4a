// Internal interface between the C ABI shim (fa_api.cu) and the kernel
// translation units. Host-only declarations; no CUDA types beyond CUtensorMap.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

struct FwdArgs {
  CUtensorMap tm_q, tm_o;  // bf16 [BH][Nq][d], box 64 x 128 x 1, 128B swizzle
  CUtensorMap tm_k, tm_v;  // bf16 [BH][Nk][d], the same boxes
  void* o;                 // bf16 [BH][Nq][d] (written by the merge kernel when the keys are split)
  float* lse;              // fp32 [BH][Nq]
  unsigned int* status;    // device error word
  int BH, H, Nq, Nk, d;
  float scale_log2;  // scale * log2(e) (8-bit inputs: times the q and k dequantisation factors)
  float o_scale;     // factor on O / l: 1, or the v dequantisation factor for 8-bit inputs
  int fp8;           // q, k, v are E4M3 codes (d = 128 only)
  int causal;        // query row i sees keys 0 .. i + Nk - Nq (needs Nq <= Nk)
  // optional per-sequence lengths, int32 [B] (padding masks): batch b has only
  // its first seq_len(seqlens_q, b, Nq) query rows and seq_len(seqlens_k, b, Nk) keys
  const int* seqlens_q;
  const int* seqlens_k;
  // dropout of P after the softmax (probability drop_p256 / 256; 0: none):
  // Philox4x32-10 round keys of the seed, the counter's fourth word
  int drop_p256;
  unsigned int drop_offset;
  unsigned int drop_rk[20];
  int head_group;    // heads per CTA scheduling group (set by launch_fwd)
  // Key ranges per query block. With n_split > 1, CTA z covers key blocks
  // [z * split_blocks, (z + 1) * split_blocks) and writes O / l (fp32) and the
  // range's logsumexp to o_part [n_split][BH][Nq][d] and lse_part
  // [n_split][BH][Nq]; a merge kernel then writes o and lse.
  int n_split, split_blocks;
  float* o_part;
  float* lse_part;
  // Test hook (fa_test_arm_fault), 0 in normal use. 1: the load warp of every
  // CTA withholds the first query tile's copy, so the MMA warp's bounded wait
  // for it expires and the CTA takes its abort path.
  int test_fault;
};

struct BwdArgs {
  // bf16, box 64 x 128 x 1, 128B swizzle: q, dO, dq over [BH][Nq][d]; k, v, dk, dv over [BH][Nk][d]
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // loads
  CUtensorMap tm_o;                     // o, loaded by the d = 64 dQ kernel, which forms D itself
  CUtensorMap tm_dq, tm_dk, tm_dv;      // stores
  const void* o;                        // bf16 [BH][Nq][d]
  const void* dO;                       // bf16 [BH][Nq][d]
  const float* lse;                     // fp32 [BH][Nq]
  float* Dsum;                          // fp32 [BH][Nq], in the caller's workspace
  unsigned int* work;                   // work counters in the caller's workspace ([0] dK/dV, [1] dQ)
  unsigned int* status;
  int BH, H, Nq, Nk, d;
  float scale, scale_log2;
  int causal;         // query row i sees keys 0 .. i + Nk - Nq (needs Nq <= Nk)
  const int* seqlens_q;  // optional per-sequence lengths, as in FwdArgs
  const int* seqlens_k;
  int drop_p256;          // dropout, as in FwdArgs (the forward's seed and offset)
  unsigned int drop_offset;
  unsigned int drop_rk[20];
  float drop_scale;       // 256 / (256 - drop_p256)
  int head_group;     // heads per CTA scheduling group of the dK/dV kernel (set by launch_bwd)
  int head_group_dq;  // the same for the dQ kernel
};

// Status bit a kernel sets when a per-sequence length lies outside [1, N]
// (or, under the causal mask, a query length exceeds its key length); the
// kernel then works with the length clamped into range.
constexpr unsigned int kStatusBadLength = 32u;

// Lengths of sequence b under the padding masks: sq query rows and sk keys,
// each lens[b] clamped to [1, N] (N without lengths), and under the causal
// mask sq cut to sk, so that every valid row sees a key. Returns true when a
// length had to be changed.
__device__ inline bool seq_lens(const int* lq, const int* lk, int b, int Nq, int Nk, bool causal, int& sq, int& sk) {
  bool bad = false;
  sq = Nq;
  sk = Nk;
  if (lq) {
    const int x = lq[b];
    sq = x < 1 ? 1 : (x > Nq ? Nq : x);
    bad |= sq != x;
  }
  if (lk) {
    const int x = lk[b];
    sk = x < 1 ? 1 : (x > Nk ? Nk : x);
    bad |= sk != x;
  }
  if (causal && sq > sk) {
    sq = sk;
    bad = true;
  }
  return bad;
}

// Forward CTA shape for head dimension d: query rows per CTA and CTAs that
// share an SM (d = 64: one 128-row tile, two CTAs per SM; else two tiles, one).
inline int fwd_rows_per_cta(int d) { return d == 64 ? 128 : 256; }
inline int fwd_ctas_per_sm(int d) { return d == 64 ? 2 : 1; }

// Heads per CTA scheduling group for a (BH x nblk) grid whose causal CTAs
// cost nblk - blk units of work plus 'overhead' units each (schedule.cu).
int pick_head_group(int BH, int nblk, bool causal, int num_sms, double overhead);

// Each returns cudaSuccess or the launch error.
cudaError_t launch_fwd(const FwdArgs& a, int num_sms, cudaStream_t stream);
// Key ranges worth splitting a forward into (1 = no split, when the query
// blocks alone fill the SMs): the fewest whose CTAs (rows_per_cta query rows
// each) fill their waves of num_slots CTAs (SMs x CTAs per SM) to 90%, each
// range at least two 128-key blocks, at most kMaxKeySplits.
constexpr int kMaxKeySplits = 32;
int pick_key_splits(int BH, int Nq, int Nk, int num_slots, int rows_per_cta);
cudaError_t launch_bwd(const BwdArgs& a, int num_sms, cudaStream_t stream);
// The persistent d = 64 forward (fa_fwd_persist.cu): whether it takes these
// arguments (d = 64, 16-bit, no padding masks, key ranges or dropout), and its launch.
bool fwd_persist_applies(const FwdArgs& a);
cudaError_t launch_fwd_persist(const FwdArgs& a, int num_sms, cudaStream_t stream);

}  // namespace fa
