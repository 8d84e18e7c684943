// api.cu -- the C ABI of libfp8attn.so (declared in include/fp8attn.h):
// argument checks, TMA tensor maps, and the launch of the persistent kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <random>
#include <vector>

#include "../../include/fp8attn.h"
#include "attn_fwd.cuh"
#include "quant.cuh"
#include "split_plan.h"

namespace {

using fa8::KParams;
using fa8::Maps;

constexpr unsigned long long kWaitLimitNs = 4000000000ull;      // 4 s per wait
constexpr unsigned long long kTestWaitLimitNs = 200000000ull;   // 0.2 s (stall test)
constexpr int kMaxDevices = 64;
// Item chunking thresholds (bytes of K and V): above kChunkAllBytes for the
// whole problem, chunks hold about kChunkBytes, half of the 129 MB L2, so
// that the two or three chunks' worth of kv heads in flight stay in L2.
constexpr size_t kChunkAllBytes = 256ull << 20;
constexpr size_t kChunkBytes = 64ull << 20;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 sm_103, 2 other
  int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Checks the current device once: sm_103 and its SM count.
int device_check(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  DeviceInfo& d = g_dev[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    st = d.state.load(std::memory_order_relaxed);
    if (st == 0) {
      int major = 0, minor = 0, n = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
      d.sms = n;
      st = (major == 10 && minor == 3) ? 1 : 2;
      d.state.store(st, std::memory_order_release);
    }
  }
  if (st != 1) return ATTN_ERR_ARCH;
  *sms = d.sms;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 4-D tensor map over a BSHD tensor: dims (D, H, S, B) innermost first; the
// box is `box_inner` elements of D, one head, `box_rows` rows of S, one batch.
int make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int D, int H,
             int S, int B, int box_inner, CUtensorMapSwizzle sw, int box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return ATTN_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize,
                           (cuuint64_t)S * H * D * esize};
  cuuint32_t box[4] = {(cuuint32_t)box_inner, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, dt, 4, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int V, int DQK, bool SPLIT = false>
int launch(const Maps& maps, const KParams& p, int sms, cudaStream_t stream) {
  using C = fa8::Cfg<V, DQK>;
  auto kern = fa8::attn_fwd_kernel<V, DQK, SPLIT>;
  // Per-device opt-in to the large dynamic shared memory carve-out.
  static std::atomic<unsigned long long> done_mask[1] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(done_mask[0].load(std::memory_order_acquire) & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    done_mask[0].fetch_or(bit, std::memory_order_acq_rel);
  }
  const int grid = p.n_units < sms ? p.n_units : sms;
  kern<<<grid, fa8::kThreads, C::kSmemAlloc, stream>>>(maps, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// A tag per call that uses a split workspace (see split_arrive): distinct
// across calls and, from a random start, across library copies in a process.
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> epoch{[] {
    std::random_device rd;
    return ((((unsigned long long)rd() << 32) ^ rd()) & ((1ull << 58) - 1)) + 1;
  }()};
  return epoch.fetch_add(1, std::memory_order_relaxed) & ((1ull << 61) - 1);
}

int run(int variant, const void* q, const void* k, const void* v, const float* dq, const float* dk,
        const float* dv, void* out, int out_dtype, float* lse, int B, int Hq, int Hkv, int S,
        int Dqk, int Dv, int causal, float softmax_scale, int flags, int* dev_status,
        void* workspace, size_t workspace_bytes, void* stream) {
  // ---- argument checks (before anything touches the device)
  if (variant < ATTN_VARIANT_LEANP || variant > ATTN_VARIANT_LEANP_A3) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_OUT_BF16 && out_dtype != ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return ATTN_ERR_INVALID_ARG;
  const bool fp8 = variant != ATTN_VARIANT_BF16;
  if (fp8 && (!dq || !dk || !dv)) return ATTN_ERR_INVALID_ARG;
  if (fp8 && ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
               reinterpret_cast<uintptr_t>(dv)) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || Dqk < 1 || Dv < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if ((flags & ATTN_FLAG_TEST_STALL_LOADS) && !dev_status) return ATTN_ERR_INVALID_ARG;
  if (flags & ~(ATTN_FLAG_TEST_STALL_LOADS | ATTN_FLAG_DESCALE_PER_BKV | ATTN_FLAG_TEST_CHUNK_UNITS))
    return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_INVALID_ARG;
  if (Dv != 128) return ATTN_ERR_UNSUPPORTED;
  if (fp8 ? (Dqk != 128 && Dqk != 192) : (Dqk != 128)) return ATTN_ERR_UNSUPPORTED;
  // index ranges: the kernel's int arithmetic covers B*Hq*ceil(S/256) items
  const long long n_qblocks = (S + 255) / 256;
  const long long n_items = (long long)B * Hq * n_qblocks;
  if (n_items > (1ll << 30) || (long long)B * S > (1ll << 31)) return ATTN_ERR_INVALID_ARG;

  int sms = 0;
  int st = device_check(&sms);
  if (st != ATTN_OK) return st;

  KParams p;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S = S;
  p.group = Hq / Hkv;
  p.n_qblocks = (int)n_qblocks;
  p.n_kv_tiles = (S + 127) / 128;
  p.n_items = (int)n_items;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt((float)Dqk);
  p.out = out;
  p.out_f32 = out_dtype == ATTN_OUT_F32;
  p.status = dev_status;
  p.flags = flags;
  p.wait_limit_ns = (flags & ATTN_FLAG_TEST_STALL_LOADS) ? kTestWaitLimitNs : kWaitLimitNs;
  // Item chunks (see decode_item): one chunk while the K and V of all
  // (batch, kv head) units take at most kChunkAllBytes; beyond that, chunks
  // of about kChunkBytes of K and V each (at least one unit).
  {
    const size_t kv_unit = (size_t)S * (size_t)(Dqk + Dv) * (size_t)(fp8 ? 1 : 2);
    const long long units = (long long)B * Hkv;
    long long g = units;
    if (flags & ATTN_FLAG_TEST_CHUNK_UNITS) {
      g = 1;
    } else if (kv_unit * (size_t)units > kChunkAllBytes) {
      g = (long long)(kChunkBytes / kv_unit);
      if (g < 1) g = 1;
      if (g > units) g = units;
    }
    p.chunk_q = (int)(g * (Hq / Hkv));
  }
  p.causal = causal;
  p.descale_per_bkv = (flags & ATTN_FLAG_DESCALE_PER_BKV) ? 1 : 0;
  p.lse = lse;
  // Split schedule: with a workspace, for the paths whose codes depend on each
  // key block alone, in the plain (unchunked) item order.
  SplitPlan plan;
  if (workspace && split_variant(variant) && p.chunk_q == B * Hq)
    plan = split_plan(B * Hq, S, causal, split_costs(variant, Dqk), sms, kSplitMaxBytes);
  if (plan.n_split_items > 0 && workspace_bytes < plan.ws_bytes) return ATTN_ERR_INVALID_ARG;
  p.split_qb = plan.split_qb;
  p.split_ns = plan.ns;
  p.n_split_items = plan.n_split_items;
  p.n_units = (int)(n_items + (long long)plan.n_split_items * (plan.ns - 1));
  p.ws = plan.n_split_items > 0 ? static_cast<unsigned char*>(workspace) : nullptr;
  p.epoch = plan.n_split_items > 0 ? next_epoch() : 0;
  const bool split = plan.n_split_items > 0;

  Maps maps;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int es = fp8 ? 1 : 2;
  const int inner = 128 / es;  // elements per 128-byte panel
  if ((st = make_map(&maps.q128, q, dt, es, Dqk, Hq, S, B, inner, CU_TENSOR_MAP_SWIZZLE_128B)))
    return st;
  if ((st = make_map(&maps.k128, k, dt, es, Dqk, Hkv, S, B, inner, CU_TENSOR_MAP_SWIZZLE_128B)))
    return st;
  if ((st = make_map(&maps.v, v, dt, es, Dv, Hkv, S, B, inner, CU_TENSOR_MAP_SWIZZLE_128B)))
    return st;
  if (Dqk == 192) {
    if ((st = make_map(&maps.q64, q, dt, es, Dqk, Hq, S, B, 64, CU_TENSOR_MAP_SWIZZLE_64B)))
      return st;
    if ((st = make_map(&maps.k64, k, dt, es, Dqk, Hkv, S, B, 64, CU_TENSOR_MAP_SWIZZLE_64B)))
      return st;
  } else {
    maps.q64 = maps.q128;
    maps.k64 = maps.k128;
  }
  // bf16 output of the FP8 paths: TMA stores in boxes of 64 columns x 32 rows
  if (fp8 && out_dtype == ATTN_OUT_BF16) {
    if ((st = make_map(&maps.o64, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Dv, Hq, S, B, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, 32)))
      return st;
  } else {
    maps.o64 = maps.v;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (split) {
    if (variant == ATTN_VARIANT_BF16) return launch<fa8::kBf16, 128, true>(maps, p, sms, s);
    if (variant == ATTN_VARIANT_LEANP)
      return Dqk == 128 ? launch<fa8::kLeanP, 128, true>(maps, p, sms, s)
                        : launch<fa8::kLeanP, 192, true>(maps, p, sms, s);
    return Dqk == 128 ? launch<fa8::kBlockExact, 128, true>(maps, p, sms, s)
                      : launch<fa8::kBlockExact, 192, true>(maps, p, sms, s);
  }
  switch (variant) {
    case ATTN_VARIANT_LEANP:
      return Dqk == 128 ? launch<fa8::kLeanP, 128>(maps, p, sms, s)
                        : launch<fa8::kLeanP, 192>(maps, p, sms, s);
    case ATTN_VARIANT_EXACT_FP8:
      return Dqk == 128 ? launch<fa8::kExactFp8, 128>(maps, p, sms, s)
                        : launch<fa8::kExactFp8, 192>(maps, p, sms, s);
    case ATTN_VARIANT_BLOCK_EXACT:
      return Dqk == 128 ? launch<fa8::kBlockExact, 128>(maps, p, sms, s)
                        : launch<fa8::kBlockExact, 192>(maps, p, sms, s);
    case ATTN_VARIANT_LEANP_A3:
      return Dqk == 128 ? launch<fa8::kLeanPA3, 128>(maps, p, sms, s)
                        : launch<fa8::kLeanPA3, 192>(maps, p, sms, s);
    default:
      return launch<fa8::kBf16, 128>(maps, p, sms, s);
  }
}

}  // namespace

extern "C" {

int attn_fwd_fp8(const void* q, const void* k, const void* v, const float* descale_q,
                 const float* descale_k, const float* descale_v, void* out, int B, int Hq,
                 int Hkv, int S, int Dqk, int Dv, int causal, void* stream) {
  return run(ATTN_VARIANT_LEANP, q, k, v, descale_q, descale_k, descale_v, out, ATTN_OUT_BF16,
             nullptr, B, Hq, Hkv, S, Dqk, Dv, causal, 0.0f, 0, nullptr, nullptr, 0, stream);
}

int attn_fwd_fp8_exact(const void* q, const void* k, const void* v, const float* descale_q,
                       const float* descale_k, const float* descale_v, void* out, int B,
                       int Hq, int Hkv, int S, int Dqk, int Dv, int causal, void* stream) {
  return run(ATTN_VARIANT_EXACT_FP8, q, k, v, descale_q, descale_k, descale_v, out,
             ATTN_OUT_BF16, nullptr, B, Hq, Hkv, S, Dqk, Dv, causal, 0.0f, 0, nullptr, nullptr, 0,
             stream);
}

int attn_fwd_bf16(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                  int S, int Dqk, int Dv, int causal, void* stream) {
  return run(ATTN_VARIANT_BF16, q, k, v, nullptr, nullptr, nullptr, out, ATTN_OUT_BF16, nullptr,
             B, Hq, Hkv, S, Dqk, Dv, causal, 0.0f, 0, nullptr, nullptr, 0, stream);
}

int attn_fwd_ex(int variant, const void* q, const void* k, const void* v, const float* descale_q,
                const float* descale_k, const float* descale_v, void* out, int out_dtype, int B,
                int Hq, int Hkv, int S, int Dqk, int Dv, int causal, float softmax_scale,
                int flags, int* dev_status, void* stream) {
  return run(variant, q, k, v, descale_q, descale_k, descale_v, out, out_dtype, nullptr, B, Hq,
             Hkv, S, Dqk, Dv, causal, softmax_scale, flags, dev_status, nullptr, 0, stream);
}

int attn_fwd_full(int variant, const void* q, const void* k, const void* v,
                  const float* descale_q, const float* descale_k, const float* descale_v,
                  void* out, int out_dtype, float* lse, int B, int Hq, int Hkv, int S, int Dqk,
                  int Dv, int causal, float softmax_scale, int flags, int* dev_status,
                  void* workspace, size_t workspace_bytes, void* stream) {
  return run(variant, q, k, v, descale_q, descale_k, descale_v, out, out_dtype, lse, B, Hq, Hkv,
             S, Dqk, Dv, causal, softmax_scale, flags, dev_status, workspace, workspace_bytes,
             stream);
}

// The split plan attn_fwd_full uses for these arguments on a GPU with `sms`
// SMs (0: the current device, which must then pass device_check).
static int plan_query(int variant, int B, int Hq, int Hkv, int S, int Dqk, int Dv, int causal,
                      int flags, int sms, SplitPlan* plan) {
  *plan = SplitPlan();
  if (variant < ATTN_VARIANT_LEANP || variant > ATTN_VARIANT_LEANP_A3) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || Dqk < 1 || Dv < 1 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (sms < 0) return ATTN_ERR_INVALID_ARG;
  const long long n_items = (long long)B * Hq * ((S + 255) / 256);
  if (n_items > (1ll << 30) || (long long)B * S > (1ll << 31)) return ATTN_ERR_INVALID_ARG;
  if (!split_variant(variant) || (flags & ATTN_FLAG_TEST_CHUNK_UNITS)) return ATTN_OK;
  // only the unchunked item order splits (see run)
  const size_t kv_unit = (size_t)S * (size_t)(Dqk + Dv) * (variant == ATTN_VARIANT_BF16 ? 2 : 1);
  if (kv_unit * (size_t)((long long)B * Hkv) > kChunkAllBytes) return ATTN_OK;
  if (sms == 0) {
    const int st = device_check(&sms);
    if (st != ATTN_OK) return st;
  }
  *plan = split_plan(B * Hq, S, causal, split_costs(variant, Dqk), sms, kSplitMaxBytes);
  return ATTN_OK;
}

int attn_workspace_size(int variant, int B, int Hq, int Hkv, int S, int Dqk, int Dv, int causal,
                        int flags, size_t* bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  SplitPlan plan;
  const int st = plan_query(variant, B, Hq, Hkv, S, Dqk, Dv, causal, flags, 0, &plan);
  if (st == ATTN_OK) *bytes = plan.ws_bytes;
  return st;
}

int attn_split_plan(int variant, int B, int Hq, int Hkv, int S, int Dqk, int Dv, int causal,
                    int flags, int sms, int* split_qb, int* ns, size_t* bytes) {
  if (!split_qb || !ns || !bytes) return ATTN_ERR_INVALID_ARG;
  *split_qb = 0;
  *ns = 1;
  *bytes = 0;
  if (sms < 1) return ATTN_ERR_INVALID_ARG;
  SplitPlan plan;
  const int st = plan_query(variant, B, Hq, Hkv, S, Dqk, Dv, causal, flags, sms, &plan);
  if (st == ATTN_OK && plan.n_split_items > 0) {
    *split_qb = plan.split_qb;
    *ns = plan.ns;
    *bytes = plan.ws_bytes;
  }
  return st;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_ARCH: return "device is not sm_103 (GB300)";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int attn_quantize_fp8(const void* x, int in_dtype, void* codes, float* descale, int B, int S,
                      int H, int D, int hadamard, void* stream) {
  if (!x || !codes || !descale) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || (hadamard != 0 && hadamard != 1)) return ATTN_ERR_INVALID_ARG;
  if (in_dtype != ATTN_IN_BF16 && in_dtype != ATTN_IN_F32) return ATTN_ERR_INVALID_ARG;
  if (D != 128 && D != 192) return ATTN_ERR_UNSUPPORTED;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
  if ((xa & 15u) != 0 || (reinterpret_cast<uintptr_t>(codes) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(descale) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  const long long n_vec = (long long)B * S * H;
  if (n_vec > (1ll << 40)) return ATTN_ERR_INVALID_ARG;
  int sms = 0;
  const int dc = device_check(&sms);
  if (dc != ATTN_OK) return dc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // a few waves of warps, each taking eight vectors at a time
  const long long warps = (n_vec + fa8::kQuantVecPerWarp - 1) / fa8::kQuantVecPerWarp;
  const long long want = (warps * 32 + fa8::kQuantThreads - 1) / fa8::kQuantThreads;
  const int grid = (int)(want < 8ll * sms ? want : 8ll * sms);
  const float norm = !hadamard ? 1.0f : (D == 192 ? 0.125f : 0.0883883476483184405501f);
  if (cudaMemsetAsync(descale, 0, sizeof(float), s) != cudaSuccess) return ATTN_ERR_CUDA;
  const bool f32 = in_dtype == ATTN_IN_F32;
  uint8_t* c = static_cast<uint8_t*>(codes);
  if (D == 128) {
    if (f32) {
      fa8::quant_amax_kernel<128, true><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale);
      fa8::quant_codes_kernel<128, true><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale, c);
    } else {
      fa8::quant_amax_kernel<128, false><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale);
      fa8::quant_codes_kernel<128, false><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale, c);
    }
  } else {
    if (f32) {
      fa8::quant_amax_kernel<192, true><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale);
      fa8::quant_codes_kernel<192, true><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale, c);
    } else {
      fa8::quant_amax_kernel<192, false><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale);
      fa8::quant_codes_kernel<192, false><<<grid, fa8::kQuantThreads, 0, s>>>(x, n_vec, hadamard, descale, c);
    }
  }
  fa8::quant_finish_kernel<<<1, 1, 0, s>>>(descale, norm);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_launches_per_call(void) { return 1; }

int attn_api_version(void) { return FP8ATTN_API_VERSION; }

int attn_debug_timeline(unsigned long long* host, int capacity, int reset) {
#ifdef FA8_TIMELINE
  constexpr int kN = 6 * 64 * 8;
  if (!host || capacity < 0) return ATTN_ERR_INVALID_ARG;
  int sms = 0;
  const int st = device_check(&sms);
  if (st != ATTN_OK) return st;
  const int n = capacity < kN ? capacity : kN;
  if (n > 0 && cudaMemcpyFromSymbol(host, fa8::fa8_timeline, sizeof(unsigned long long) * n) !=
                   cudaSuccess)
    return ATTN_ERR_CUDA;
  if (reset) {
    static const unsigned long long zeros[kN] = {};
    if (cudaMemcpyToSymbol(fa8::fa8_timeline, zeros, sizeof zeros) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
#else
  (void)host, (void)capacity, (void)reset;
  return ATTN_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"

// ------------------------------------------------------------ no-alloc entry
// attn_fwd_fp8_noalloc: attn_fwd_fp8 with the split schedule of attn_fwd_full
// for callers that cannot allocate device memory.  Some code may not call
// cudaMalloc: a plugin or runtime that owns every device allocation through
// its own allocator, a real-time or inference loop that forbids allocations
// after start-up (an allocation can synchronise the device and stall other
// streams), or code that runs with a fixed memory budget.  Such callers can
// still pass inputs and outputs, but not a workspace, so the split schedule
// takes its scratch from this array: file-scope device memory that the driver
// sets aside when the library's module loads, on every GPU that loads it, and
// keeps until the process exits.  The split schedule tags its counters with a
// per-call number, so nothing in the array has to start at zero and nothing
// is cleared between calls; every call shares the array, so calls that
// overlap on the GPU (different streams) race on it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// The device address of g_noalloc_scratch on the current device.  In host
// code the array's name stands for a host-side shadow, not device memory, so
// the address comes from cudaGetSymbolAddress, once per device, with that
// device current.
int noalloc_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_fp8_noalloc(const void* q, const void* k, const void* v,
                                    const float* descale_q, const float* descale_k,
                                    const float* descale_v, void* out, int B, int Hq, int Hkv,
                                    int S, int Dqk, int Dv, int causal, void* stream) {
  // the schedule attn_fwd_full would choose with a workspace, and its scratch
  size_t need = 0;
  int st = attn_workspace_size(ATTN_VARIANT_LEANP, B, Hq, Hkv, S, Dqk, Dv, causal, 0, &need);
  if (st != ATTN_OK) return st;
  if (need > (size_t)ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != ATTN_OK) return st;
  return run(ATTN_VARIANT_LEANP, q, k, v, descale_q, descale_k, descale_v, out, ATTN_OUT_BF16,
             nullptr, B, Hq, Hkv, S, Dqk, Dv, causal, 0.0f, 0, nullptr, need ? scratch : nullptr,
             need ? (size_t)ATTN_NOALLOC_SCRATCH_BYTES : 0, stream);
}
