// C ABI of the attention library (declared in include/fa.h): argument
// checks, TMA tensor-map encoding, and kernel launches. Nothing here
// allocates device memory; the only device state the library owns is one
// error word per device, a file-scope __device__ variable.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "philox.cuh"

namespace {

__device__ unsigned int g_fa_device_status = 0;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  bool supported = false;
  unsigned int* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int fail_launch() { return FA_ERR_LAUNCH; }

// Fault armed by fa_test_arm_fault for the next forward launch (0: none).
std::atomic<int> g_test_fault{0};

// Per-device facts, looked up once per device with that device current.
int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail_launch();
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail_launch();
    di.supported = (major == 10 && minor == 3);  // the kernels are built for sm_103a only
    di.num_sms = sms;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_device_status) != cudaSuccess) return fail_launch();
    di.status = static_cast<unsigned int*>(p);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return fail_launch();
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    di.ready = true;
  }
  if (!di.supported) return FA_ERR_UNSUPPORTED;
  *out = &di;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const int* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }  // (NULL passes)

int check_shape(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long total = (long long)B * H * N * d;
  if ((long long)B * H > INT32_MAX || total >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Tensor map over a contiguous [BH][N][d] tensor, boxes of box_x columns by
// box_rows rows of one head, 128-byte swizzle (box_x * elem == 128 bytes).
bool encode_3d_uncached(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, int elem, int BH, int N, int d,
                        int box_x, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * elem, (cuuint64_t)N * d * elem};
  cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, dtype, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Encoded tensor maps, keyed by everything the encoding depends on: a map
// holds only the base address and the geometry, so an entry stays valid for
// any later buffer at that address with that shape and type (a freed and
// reused address with another shape is simply another key). A small set-
// associative table: 64 sets of 4 ways, least recently used way replaced.
struct MapKey {
  const void* base;
  int dev, dtype, elem, BH, N, d, box_x, box_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && dev == o.dev && dtype == o.dtype && elem == o.elem && BH == o.BH && N == o.N &&
           d == o.d && box_x == o.box_x && box_rows == o.box_rows;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  unsigned long long used;  // 0: empty
};
constexpr int kMapSets = 64, kMapWays = 4;
MapEntry g_maps[kMapSets][kMapWays];
unsigned long long g_map_clock = 0;
std::mutex g_map_mu;

int map_set(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) >> 8;
  h ^= (uint64_t)(unsigned)k.N * 0x9E3779B97F4A7C15ull;
  h ^= (uint64_t)(unsigned)k.BH * 0xC2B2AE3D27D4EB4Full;
  h ^= (uint64_t)(unsigned)(k.d + 131 * k.box_x + 17 * k.dtype + 7 * k.dev);
  h ^= h >> 29;
  return (int)(h % kMapSets);
}

bool encode_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, int elem, int BH, int N, int d,
               int box_x, int box_rows) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const MapKey key{base, dev, (int)dtype, elem, BH, N, d, box_x, box_rows};
  MapEntry* set = g_maps[map_set(key)];
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int w = 0; w < kMapWays; ++w)
      if (set[w].used && set[w].key == key) {
        set[w].used = ++g_map_clock;
        *m = set[w].map;
        return true;
      }
  }
  if (!encode_3d_uncached(m, base, dtype, elem, BH, N, d, box_x, box_rows)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  int victim = 0;
  for (int w = 1; w < kMapWays; ++w)
    if (set[w].used < set[victim].used) victim = w;
  set[victim].key = key;
  set[victim].map = *m;
  set[victim].used = ++g_map_clock;
  return true;
}

constexpr double kLog2e = 1.4426950408889634074;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The backward of every entry point: arguments validated, then the kernels (launch_bwd).
int bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
               void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
               const int* seqlens_q, const int* seqlens_k, int p256, unsigned long long seed, unsigned int offset,
               void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int st = check_shape(B, H, Nq, d, scale);
  if (st == FA_OK) st = check_shape(B, H, Nk, d, scale);
  if (st != FA_OK) return st;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;  // the first rows would see no key
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned4(seqlens_q) || !aligned4(seqlens_k))
    return FA_ERR_MISALIGNED;
  const size_t need = fa_bwd_kv_workspace_bytes(B, H, Nq, Nk, d);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FA_ERR_WORKSPACE;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  const int BH = B * H;
  fa::BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.Dsum = static_cast<float*>(workspace);
  a.work = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + (need - 256));
  if (!encode_3d(&a.tm_q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nq, d, 64, 128) ||
      !encode_3d(&a.tm_do, dO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nq, d, 64, 128) ||
      !encode_3d(&a.tm_o, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nq, d, 64, 128) ||
      !encode_3d(&a.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nk, d, 64, 128) ||
      !encode_3d(&a.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nk, d, 64, 128) ||
      !encode_3d(&a.tm_dq, dq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nq, d, 64, 128) ||
      !encode_3d(&a.tm_dk, dk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nk, d, 64, 128) ||
      !encode_3d(&a.tm_dv, dv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nk, d, 64, 128))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.status = di->status;
  a.BH = BH;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.scale = scale;
  a.scale_log2 = (float)((double)scale * kLog2e);
  a.causal = causal ? 1 : 0;
  a.seqlens_q = seqlens_q;
  a.seqlens_k = seqlens_k;
  a.drop_p256 = p256;
  a.drop_offset = offset;
  a.drop_scale = (float)(256.0 / (256.0 - p256));
  fa::philox::round_keys(seed, a.drop_rk);
  return fa::launch_bwd(a, di->num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, void* stream) {
  return fa_fwd_kv(q, k, v, o, lse, B, H, N, N, d, scale, causal, nullptr, nullptr, nullptr, 0, stream);
}

size_t fa_fwd_kv_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (check_shape(B, H, Nq, d, 1.0f) != FA_OK || check_shape(B, H, Nk, d, 1.0f) != FA_OK) return 0;
  DeviceInfo* di = nullptr;
  if (device_info(&di) != FA_OK) return 0;
  const int n = fa::pick_key_splits(B * H, Nq, Nk, di->num_sms * fa::fwd_ctas_per_sm(d), fa::fwd_rows_per_cta(d));
  if (n <= 1) return 0;
  const size_t rows = (size_t)n * B * H * Nq;
  return align256(rows * d * sizeof(float)) + align256(rows * sizeof(float));
}

int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk, int d,
              float scale, int causal, const int* seqlens_q, const int* seqlens_k, void* workspace,
              size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  int st = check_shape(B, H, Nq, d, scale);
  if (st == FA_OK) st = check_shape(B, H, Nk, d, scale);
  if (st != FA_OK) return st;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;  // the first rows would see no key
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (workspace && !aligned16(workspace)) || !aligned4(seqlens_q) || !aligned4(seqlens_k))
    return FA_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const int BH = B * H;
  if (!encode_3d(&a.tm_q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nq, d, 64, 128) ||
      !encode_3d(&a.tm_o, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nq, d, 64, 128) ||
      !encode_3d(&a.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nk, d, 64, 128) ||
      !encode_3d(&a.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, Nk, d, 64, 128))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.lse = lse;
  a.status = di->status;
  a.BH = BH;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.scale_log2 = (float)((double)scale * kLog2e);
  a.o_scale = 1.0f;
  a.causal = causal ? 1 : 0;
  a.seqlens_q = seqlens_q;
  a.seqlens_k = seqlens_k;
  // Key ranges: as many as help fill the GPU and fit the caller's workspace
  // (none without one); every range non-empty.
  const int nkv = (Nk + 127) / 128;
  int n = workspace ? fa::pick_key_splits(BH, Nq, Nk, di->num_sms * fa::fwd_ctas_per_sm(d), fa::fwd_rows_per_cta(d))
                    : 1;
  for (; n > 1; --n) {
    const size_t rows = (size_t)n * BH * Nq;
    if (align256(rows * d * sizeof(float)) + align256(rows * sizeof(float)) <= workspace_bytes) break;
  }
  a.split_blocks = (nkv + n - 1) / n;
  a.n_split = (nkv + a.split_blocks - 1) / a.split_blocks;
  if (a.n_split > 1) {
    const size_t rows = (size_t)a.n_split * BH * Nq;
    a.o_part = static_cast<float*>(workspace);
    a.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(rows * d * sizeof(float)));
  }
  a.test_fault = g_test_fault.exchange(0);
  return fa::launch_fwd(a, di->num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, float descale_q, float descale_k, float descale_v,
               void* o, float* lse, int B, int H, int N, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  int st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  const float desc[3] = {descale_q, descale_k, descale_v};
  for (float x : desc)
    if (!(x > 0.0f) || !std::isfinite(x)) return FA_ERR_INVALID_ARG;
  const float scale_log2 = (float)((double)scale * (double)descale_q * (double)descale_k * kLog2e);
  if (!std::isfinite(scale_log2) || !(scale_log2 > 0.0f)) return FA_ERR_INVALID_ARG;  // over- or underflow
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const int BH = B * H;
  // E4M3 rows of 128 bytes: one 128 x 128-byte box per tile
  if (!encode_3d(&a.tm_q, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, BH, N, d, 128, 128) ||
      !encode_3d(&a.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, BH, N, d, 128, 128) ||
      !encode_3d(&a.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, BH, N, d, 128, 128) ||
      !encode_3d(&a.tm_o, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, d, 64, 128))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.lse = lse;
  a.status = di->status;
  a.BH = BH;
  a.H = H;
  a.Nq = N;
  a.Nk = N;
  a.d = d;
  a.scale_log2 = scale_log2;
  a.o_scale = descale_v;
  a.fp8 = 1;
  a.causal = causal ? 1 : 0;
  a.split_blocks = (N + 127) / 128;
  a.n_split = 1;
  a.test_fault = g_test_fault.exchange(0);
  return fa::launch_fwd(a, di->num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   float scale, int causal, int p256, unsigned long long seed, unsigned int offset, void* stream) {
  if (!q || !k || !v || !o || !lse || p256 < 0 || p256 > 255) return FA_ERR_INVALID_ARG;
  int st = check_shape(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  fa::FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const int BH = B * H;
  if (!encode_3d(&a.tm_q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, d, 64, 128) ||
      !encode_3d(&a.tm_o, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, d, 64, 128) ||
      !encode_3d(&a.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, d, 64, 128) ||
      !encode_3d(&a.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, BH, N, d, 64, 128))
    return FA_ERR_LAUNCH;
  a.o = o;
  a.lse = lse;
  a.status = di->status;
  a.BH = BH;
  a.H = H;
  a.Nq = N;
  a.Nk = N;
  a.d = d;
  a.scale_log2 = (float)((double)scale * kLog2e);
  a.o_scale = (float)(256.0 / (256.0 - p256));  // kept elements carry 1 / (1 - p)
  a.causal = causal ? 1 : 0;
  a.drop_p256 = p256;
  a.drop_offset = offset;
  fa::philox::round_keys(seed, a.drop_rk);
  a.split_blocks = (N + 127) / 128;
  a.n_split = 1;
  a.test_fault = g_test_fault.exchange(0);
  return fa::launch_fwd(a, di->num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) { return fa_bwd_kv_workspace_bytes(B, H, N, N, d); }

size_t fa_bwd_kv_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (check_shape(B, H, Nq, d, 1.0f) != FA_OK || check_shape(B, H, Nk, d, 1.0f) != FA_OK) return 0;
  const size_t rows = (size_t)B * H * Nq;
  return align256(rows * sizeof(float)) + 256;  // D, then the kernels' work counters
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* workspace,
           size_t workspace_bytes, void* stream) {
  return fa_bwd_kv(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, scale, causal, nullptr, nullptr, workspace,
                   workspace_bytes, stream);
}

int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int p256,
                   unsigned long long seed, unsigned int offset, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (p256 < 0 || p256 > 255) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, N, d, scale, causal, nullptr, nullptr, p256, seed,
                    offset, workspace, workspace_bytes, stream);
}

int fa_bwd_kv(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
              void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
              const int* seqlens_q, const int* seqlens_k, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, seqlens_q, seqlens_k, 0, 0, 0,
                    workspace, workspace_bytes, stream);
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or device";
    case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FA_ERR_LAUNCH: return "CUDA launch or query failed";
    case FA_ERR_TIMEOUT: return "a kernel wait timed out";
    default: return "unknown status";
  }
}

int fa_test_arm_fault(int kind) {
  if (kind < 0 || kind > 1) return FA_ERR_INVALID_ARG;
  g_test_fault.store(kind);
  return FA_OK;
}

int fa_device_status(int reset) {
  DeviceInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_LAUNCH;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_fa_device_status, sizeof(word)) != cudaSuccess) return FA_ERR_LAUNCH;
  if (reset && word) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_device_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  if (word & ~fa::kStatusBadLength) return FA_ERR_TIMEOUT;
  return word ? FA_ERR_INVALID_ARG : FA_OK;
}

}  // extern "C"
