// rf_api.cu -- the C ABI of librf.so (declared in include/rf.h).
//
// Host code only: argument validation, kernel selection and launch.  Every
// check runs before anything is enqueued; a failing check returns a status and
// records a message for rf_last_error().  The device-side status word that
// kernels set when a bounded wait runs out lives here.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "rf.h"
#include "rf_internal.h"

namespace {

thread_local char g_last_error[512] = "";

rf_status_t fail(rf_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

const char* dt_name(rf_dtype_t d) {
  switch (d) {
    case RF_F32: return "f32";
    case RF_F16: return "f16";
    case RF_BF16: return "bf16";
  }
  return "?";
}

bool valid_dtype(rf_dtype_t d) { return d == RF_F32 || d == RF_F16 || d == RF_BF16; }

// Rejects pointers the current device cannot use as device memory (host or
// unregistered memory, or another device's memory).  Runs after the pure host
// checks, so argument errors are reported without touching CUDA.
rf_status_t check_dev_ptr(const void* p, const char* name) {
  if (p == nullptr) return RF_OK;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RF_ERR_INVALID_ARG, "%s: cannot query pointer (%s)", name, cudaGetErrorString(e));
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return fail(RF_ERR_INVALID_ARG, "%s is not device memory (pass a device pointer)", name);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(RF_ERR_CUDA, "cudaGetDevice failed");
  }
  if (a.type == cudaMemoryTypeDevice && a.device != dev)
    return fail(RF_ERR_INVALID_ARG, "%s lives on device %d, current device is %d", name, a.device, dev);
  return RF_OK;
}

#define RF_TRY(expr)                   \
  do {                                 \
    rf_status_t _st = (expr);          \
    if (_st != RF_OK) return _st;      \
  } while (0)

rf_status_t launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RF_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  }
  g_last_error[0] = '\0';
  return RF_OK;
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace

// Device status word: set (atomicOr) by a kernel whose bounded wait ran out.
__device__ unsigned int g_rf_status;

namespace rf {

unsigned* device_status_ptr() {
  static std::mutex mu;
  static unsigned* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rf_status) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}

int device_sm_count() {
  static std::mutex mu;
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    counts[dev] = n;
  }
  return counts[dev];
}

long long device_l2_bytes() {
  static std::mutex mu;
  static long long bytes[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (bytes[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    bytes[dev] = n;
  }
  return bytes[dev];
}

bool encode_tma_3d_16bit(void* tmap_out, const void* base, uint64_t inner, uint64_t rows,
                         uint64_t outer, uint32_t box_rows, cudaError_t* err) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  if (encode == nullptr) {
    *err = cudaErrorNotSupported;
    return false;
  }
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * 2, inner * 2 * rows};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(reinterpret_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                      const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = cudaErrorInvalidValue;
    return false;
  }
  return true;
}

}  // namespace rf

extern "C" {

const char* rf_last_error(void) { return g_last_error; }

int rf_version(void) { return RF_VERSION; }

int rf_checks_enabled(void) {
#ifdef RF_CHECKS
  return 1;
#else
  return 0;
#endif
}

rf_status_t rf_device_status(void* stream, int clear) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RF_ERR_CUDA, "stream synchronise failed: %s", cudaGetErrorString(e));
  }
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_rf_status, sizeof(v));
  if (e == cudaSuccess && clear) {
    unsigned z = 0;
    e = cudaMemcpyToSymbol(g_rf_status, &z, sizeof(z));
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RF_ERR_CUDA, "status word access failed: %s", cudaGetErrorString(e));
  }
  if (v & 2u) return fail(RF_ERR_CHECK, "a device-side index check failed (code 0x%x)", v);
  if (v != 0) return fail(RF_ERR_TIMEOUT, "a device-side bounded wait ran out (code 0x%x)", v);
  g_last_error[0] = '\0';
  return RF_OK;
}

}  // extern "C"

namespace {

struct RopeOpt {
  int mode = 0;
  float base = 0.f;
  int pos = 0;
};

rf_status_t attn_impl(const char* name, const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal, int window,
                      const float* alibi, void* ws, size_t ws_bytes, rf_dtype_t dtype, void* stream,
                      const RopeOpt& rope = RopeOpt{}) {
  if (!q || !k || !v || !o) return fail(RF_ERR_INVALID_ARG, "%s: q, k, v and o must be non-null", name);
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || D <= 0)
    return fail(RF_ERR_INVALID_ARG, "%s: sizes must be positive (B=%d Hq=%d Hkv=%d Nq=%d Nk=%d D=%d)", name, B, Hq,
                Hkv, Nq, Nk, D);
  if (Hq % Hkv != 0) return fail(RF_ERR_INVALID_ARG, "%s: Hq=%d is not a multiple of Hkv=%d", name, Hq, Hkv);
  if (!(scale > 0.0f) || !std::isfinite(scale))
    return fail(RF_ERR_INVALID_ARG, "%s: scale must be finite and positive", name);
  if (!valid_dtype(dtype)) return fail(RF_ERR_INVALID_ARG, "%s: unknown dtype %d", name, int(dtype));
  if (window < 0) return fail(RF_ERR_INVALID_ARG, "%s: window must be >= 0", name);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(ws))
    return fail(RF_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", name);
  if ((reinterpret_cast<uintptr_t>(alibi) & 3u) != 0)
    return fail(RF_ERR_INVALID_ARG, "%s: alibi_slopes must be 4-byte aligned", name);
  if (causal && Nq != Nk)
    return fail(RF_ERR_UNSUPPORTED, "%s: causal mask requires Nq == Nk (got %d, %d)", name, Nq, Nk);
  if (!causal && (window > 0 || alibi))
    return fail(RF_ERR_UNSUPPORTED, "%s: a sliding window and ALiBi need the causal mask", name);
  if (rope.mode < 0 || rope.mode > 2) return fail(RF_ERR_INVALID_ARG, "%s: rope=%d must be 0, 1 or 2", name, rope.mode);
  if (rope.mode) {
    if (rope.pos < 0) return fail(RF_ERR_INVALID_ARG, "%s: rope_pos_offset must be >= 0", name);
    if (!std::isfinite(rope.base) || rope.base < 0.0f || rope.base == 1.0f)
      return fail(RF_ERR_INVALID_ARG, "%s: rope_base must be finite, positive and not 1 (0 = 10000)", name);
    if (dtype == RF_F32)
      return fail(RF_ERR_UNSUPPORTED, "%s: rotary embedding inside the kernel needs f16 or bf16", name);
    if (alibi) return fail(RF_ERR_UNSUPPORTED, "%s: rotary embedding with ALiBi is not built", name);
    if (static_cast<long long>(rope.pos) + (Nq > Nk ? Nq : Nk) > (1LL << 24))
      return fail(RF_ERR_UNSUPPORTED, "%s: rotary positions reach past 2^24", name);
  }
  if (dtype == RF_F32) {
    if (D % 4 != 0 || D > 128)
      return fail(RF_ERR_UNSUPPORTED, "%s: f32 path needs D %% 4 == 0 and D <= 128 (D=%d)", name, D);
  } else if (D != 64 && D != 128) {
    return fail(RF_ERR_UNSUPPORTED, "%s: %s path supports D in {64, 128} (D=%d)", name, dt_name(dtype), D);
  }
  RF_TRY(check_dev_ptr(q, "q"));
  RF_TRY(check_dev_ptr(k, "k"));
  RF_TRY(check_dev_ptr(v, "v"));
  RF_TRY(check_dev_ptr(o, "o"));
  RF_TRY(check_dev_ptr(lse, "lse"));
  RF_TRY(check_dev_ptr(alibi, "alibi_slopes"));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int sms = 0;
  if (ws && dtype != RF_F32 && !causal) {  // the split tail needs the workspace it is sized for
    sms = rf::device_sm_count();
    if (sms <= 0) return fail(RF_ERR_CUDA, "%s: cannot query the multiprocessor count", name);
    const size_t need = rf::attn_tc_workspace_bytes(B, Hq, Nq, Nk, D, causal, sms);
    if (ws_bytes < need)
      return fail(RF_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", name, need, ws_bytes);
    RF_TRY(check_dev_ptr(ws, "workspace"));
  } else if (dtype != RF_F32 && causal && window > 0 && window <= rf::kWindowPersistMax && D == 64 && !rope.mode) {
    // the persistent windowed kernel
    sms = rf::device_sm_count();
  }
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "%s: cannot resolve the device status word", name);
  if (dtype == RF_F32)
    return launched(rf::launch_attn_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                        static_cast<const float*>(v), static_cast<float*>(o), lse, B, Hq, Hkv, Nq, Nk,
                                        D, scale, causal, window, alibi, st, s),
                    name);
  const double rope_base = rope.base == 0.0f ? 10000.0 : static_cast<double>(rope.base);
  return launched(rf::launch_attn_tc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi,
                                     static_cast<rf::Dt>(dtype), st, sms > 0 ? ws : nullptr, sms, rope.mode,
                                     rope_base, rope.pos, s),
                  name);
}

}  // namespace

extern "C" {

rf_status_t rf_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Nq, int Nk, int D, float scale, int causal, rf_dtype_t dtype, void* stream) {
  return attn_impl("rf_attn_fwd", q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal ? 1 : 0, 0, nullptr, nullptr,
                   0, dtype, stream);
}

rf_status_t rf_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                           int Hkv, int Nq, int Nk, int D, float scale, const rf_attn_opts_t* opts,
                           rf_dtype_t dtype, void* stream) {
  const int causal = opts ? (opts->causal ? 1 : 0) : 0;
  const int window = opts ? opts->window : 0;
  const float* alibi = opts ? opts->alibi_slopes : nullptr;
  void* ws = opts ? opts->workspace : nullptr;
  const size_t ws_bytes = opts ? opts->workspace_bytes : 0;
  RopeOpt rope;
  if (opts) {
    rope.mode = opts->rope;
    rope.base = opts->rope_base;
    rope.pos = opts->rope_pos_offset;
  }
  return attn_impl("rf_attn_fwd_ex", q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, alibi, ws,
                   ws_bytes, dtype, stream, rope);
}

size_t rf_attn_fwd_workspace_bytes(int B, int Hq, int Nq, int Nk, int D, int causal, rf_dtype_t dtype) {
  if (B <= 0 || Hq <= 0 || Nq <= 0 || Nk <= 0 || D <= 0 || !valid_dtype(dtype)) return static_cast<size_t>(-1);
  if (causal || dtype == RF_F32) return 0;
  if (D != 64 && D != 128) return static_cast<size_t>(-1);
  const int sms = rf::device_sm_count();
  if (sms <= 0) return static_cast<size_t>(-1);
  return rf::attn_tc_workspace_bytes(B, Hq, Nq, Nk, D, causal, sms);
}

size_t rf_attn_decode_splitkv_workspace_bytes(int B, int Hq, int D, int num_splits) {
  if (B <= 0 || Hq <= 0 || D <= 0 || num_splits <= 0) return 0;
  size_t rows = size_t(B) * size_t(Hq);
  return align256(rows * size_t(num_splits) * size_t(D) * 4) + rows * size_t(num_splits) * 4;
}

rf_status_t rf_attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* o,
                                   float* lse, void* workspace, size_t workspace_bytes, int B, int Hq,
                                   int Hkv, int L, int D, int num_splits, float scale,
                                   rf_dtype_t dtype, void* stream) {
  if (!q || !k_cache || !v_cache || !o || !workspace)
    return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: q, k_cache, v_cache, o and workspace must be non-null");
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || D <= 0 || num_splits <= 0)
    return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: sizes must be positive");
  if (Hq % Hkv != 0)
    return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (!(scale > 0.0f) || !std::isfinite(scale))
    return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: scale must be finite and positive");
  if (!valid_dtype(dtype)) return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: unknown dtype %d", int(dtype));
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse))
    return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: workspace must be 256-byte aligned");
  size_t need = rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, num_splits);
  if (workspace_bytes < need)
    return fail(RF_ERR_INVALID_ARG, "rf_attn_decode_splitkv: workspace too small (%zu < %zu bytes)",
                workspace_bytes, need);
  if (dtype == RF_F32) return fail(RF_ERR_UNSUPPORTED, "rf_attn_decode_splitkv: f32 is not supported");
  if (D != 64 && D != 128)
    return fail(RF_ERR_UNSUPPORTED, "rf_attn_decode_splitkv: D must be 64 or 128 (D=%d)", D);
  if (Hq / Hkv > 8)
    return fail(RF_ERR_UNSUPPORTED, "rf_attn_decode_splitkv: at most 8 query heads per kv head (got %d)", Hq / Hkv);
  if (num_splits > 256)
    return fail(RF_ERR_UNSUPPORTED, "rf_attn_decode_splitkv: num_splits must be <= 256 (got %d)", num_splits);
  RF_TRY(check_dev_ptr(q, "q"));
  RF_TRY(check_dev_ptr(k_cache, "k_cache"));
  RF_TRY(check_dev_ptr(v_cache, "v_cache"));
  RF_TRY(check_dev_ptr(o, "o"));
  RF_TRY(check_dev_ptr(lse, "lse"));
  RF_TRY(check_dev_ptr(workspace, "workspace"));
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_attn_decode_splitkv: cannot resolve the device status word");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  size_t rows = size_t(B) * size_t(Hq);
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             align256(rows * size_t(num_splits) * size_t(D) * 4));
  rf_status_t r = launched(rf::launch_decode_split(q, k_cache, v_cache, o_part, lse_part, B, Hq, Hkv, L,
                                                   D, num_splits, scale, static_cast<rf::Dt>(dtype), st, s),
                           "rf_attn_decode_splitkv(split)");
  if (r != RF_OK) return r;
  return launched(rf::launch_lse_merge(o_part, lse_part, o, lse, int(rows), num_splits, D,
                                       static_cast<rf::Dt>(dtype), st, s, /*after_split=*/true),
                  "rf_attn_decode_splitkv(merge)");
}

rf_status_t rf_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse, int rows,
                         int num_splits, int D, rf_dtype_t out_dtype, void* stream) {
  if (!o_part || !lse_part || !o) return fail(RF_ERR_INVALID_ARG, "rf_lse_merge: o_part, lse_part and o must be non-null");
  if (rows <= 0 || num_splits <= 0 || D <= 0)
    return fail(RF_ERR_INVALID_ARG, "rf_lse_merge: sizes must be positive");
  if (!valid_dtype(out_dtype)) return fail(RF_ERR_INVALID_ARG, "rf_lse_merge: unknown dtype %d", int(out_dtype));
  if (!aligned16(o_part) || !aligned16(o))
    return fail(RF_ERR_INVALID_ARG, "rf_lse_merge: o_part and o must be 16-byte aligned");
  if (D % 4 != 0 || D > 512) return fail(RF_ERR_UNSUPPORTED, "rf_lse_merge: D must be a multiple of 4, <= 512");
  if (num_splits > 256) return fail(RF_ERR_UNSUPPORTED, "rf_lse_merge: num_splits must be <= 256");
  RF_TRY(check_dev_ptr(o_part, "o_part"));
  RF_TRY(check_dev_ptr(lse_part, "lse_part"));
  RF_TRY(check_dev_ptr(o, "o"));
  RF_TRY(check_dev_ptr(lse, "lse"));
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_lse_merge: cannot resolve the device status word");
  return launched(rf::launch_lse_merge(o_part, lse_part, o, lse, rows, num_splits, D,
                                       static_cast<rf::Dt>(out_dtype), st, static_cast<cudaStream_t>(stream)),
                  "rf_lse_merge");
}

rf_status_t rf_layernorm_fused(const void* x, const void* residual, const void* gamma, const void* beta,
                               void* out, void* residual_out, int rows, int cols, float eps,
                               rf_dtype_t dtype, void* stream) {
  if (!x || !out) return fail(RF_ERR_INVALID_ARG, "rf_layernorm_fused: x and out must be non-null");
  if (rows <= 0 || cols <= 0) return fail(RF_ERR_INVALID_ARG, "rf_layernorm_fused: sizes must be positive");
  if (!(eps >= 0.0f) || !std::isfinite(eps))
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_fused: eps must be finite and >= 0");
  if (!valid_dtype(dtype)) return fail(RF_ERR_INVALID_ARG, "rf_layernorm_fused: unknown dtype %d", int(dtype));
  if (!aligned16(x) || !aligned16(residual) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out) ||
      !aligned16(residual_out))
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_fused: pointers must be 16-byte aligned");
  int vec = dtype == RF_F32 ? 4 : 8;
  if (cols % vec != 0)
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_fused: cols=%d must be a multiple of %d for %s", cols, vec,
                dt_name(dtype));
  if (cols > rf::layernorm_max_cols(static_cast<rf::Dt>(dtype)))
    return fail(RF_ERR_UNSUPPORTED, "rf_layernorm_fused: cols=%d exceeds %d", cols,
                rf::layernorm_max_cols(static_cast<rf::Dt>(dtype)));
  RF_TRY(check_dev_ptr(x, "x"));
  RF_TRY(check_dev_ptr(residual, "residual"));
  RF_TRY(check_dev_ptr(gamma, "gamma"));
  RF_TRY(check_dev_ptr(beta, "beta"));
  RF_TRY(check_dev_ptr(out, "out"));
  RF_TRY(check_dev_ptr(residual_out, "residual_out"));
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_layernorm_fused: cannot resolve the device status word");
  return launched(rf::launch_layernorm(x, residual, gamma, beta, out, residual_out, rows, cols, eps,
                                       static_cast<rf::Dt>(dtype), st, static_cast<cudaStream_t>(stream)),
                  "rf_layernorm_fused");
}

rf_status_t rf_rope_qk(const void* q, const void* k, void* q_out, void* k_out, int B, int Hq, int Hkv, int N, int D,
                       float base, int pos_offset, rf_dtype_t dtype, void* stream) {
  if (!q || !q_out) return fail(RF_ERR_INVALID_ARG, "rf_rope_qk: q and q_out must be non-null");
  if ((k == nullptr) != (k_out == nullptr))
    return fail(RF_ERR_INVALID_ARG, "rf_rope_qk: k and k_out must both be given or both be null");
  if (B <= 0 || Hq <= 0 || N <= 0 || D <= 0 || (k && Hkv <= 0))
    return fail(RF_ERR_INVALID_ARG, "rf_rope_qk: sizes must be positive (B=%d Hq=%d Hkv=%d N=%d D=%d)", B, Hq, Hkv,
                N, D);
  if (!(base > 0.0f) || !std::isfinite(base) || base == 1.0f)
    return fail(RF_ERR_INVALID_ARG, "rf_rope_qk: base must be finite, positive and not 1");
  if (pos_offset < 0) return fail(RF_ERR_INVALID_ARG, "rf_rope_qk: pos_offset must be >= 0");
  if (!valid_dtype(dtype)) return fail(RF_ERR_INVALID_ARG, "rf_rope_qk: unknown dtype %d", int(dtype));
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_out) || !aligned16(k_out))
    return fail(RF_ERR_INVALID_ARG, "rf_rope_qk: pointers must be 16-byte aligned");
  if (dtype == RF_F32) return fail(RF_ERR_UNSUPPORTED, "rf_rope_qk: fp32 is not supported (f16, bf16)");
  if (D != 64 && D != 128 && D != 256) return fail(RF_ERR_UNSUPPORTED, "rf_rope_qk: D=%d (64, 128, 256)", D);
  if (static_cast<long long>(pos_offset) + N > (1LL << 24))
    return fail(RF_ERR_UNSUPPORTED, "rf_rope_qk: positions reach %lld, past 2^24",
                static_cast<long long>(pos_offset) + N);
  // one CTA indexes (B*Hq + B*Hkv) rows x 8 positions x D/16 chunk pairs in 32 bits (with headroom)
  if ((static_cast<long long>(B) * Hq + static_cast<long long>(B) * Hkv) * 8 * (D / 16) > 0x7fff0000LL)
    return fail(RF_ERR_UNSUPPORTED, "rf_rope_qk: B*(Hq+Hkv) too large");
  RF_TRY(check_dev_ptr(q, "q"));
  RF_TRY(check_dev_ptr(k, "k"));
  RF_TRY(check_dev_ptr(q_out, "q_out"));
  RF_TRY(check_dev_ptr(k_out, "k_out"));
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_rope_qk: cannot resolve the device status word");
  return launched(rf::launch_rope_qk(q, k, q_out, k_out, B * Hq, k ? B * Hkv : 0, N, D, static_cast<double>(base),
                                     pos_offset, static_cast<rf::Dt>(dtype), st, static_cast<cudaStream_t>(stream)),
                  "rf_rope_qk");
}

rf_status_t rf_selftest_wait_timeout(unsigned timeout_us, void* stream) {
  if (timeout_us == 0 || timeout_us > 1000000u)
    return fail(RF_ERR_INVALID_ARG, "rf_selftest_wait_timeout: timeout_us must be in [1, 1000000]");
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_selftest_wait_timeout: cannot resolve the device status word");
  return launched(rf::launch_wait_timeout_selftest(uint64_t(timeout_us) * 1000u, st, nullptr,
                                                   static_cast<cudaStream_t>(stream)),
                  "rf_selftest_wait_timeout");
}

rf_status_t rf_selftest_check(void* stream) {
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_selftest_check: cannot resolve the device status word");
  return launched(rf::launch_check_selftest(st, static_cast<cudaStream_t>(stream)), "rf_selftest_check");
}

rf_status_t rf_softmax_xent(const void* logits, const long long* targets, float* loss, float* lse, void* grad,
                            int rows, int vocab, long long ignore_index, rf_dtype_t dtype, void* stream) {
  if (!logits || !targets || !loss)
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent: logits, targets and loss must be non-null");
  if (rows <= 0 || vocab <= 0) return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent: sizes must be positive");
  if (!valid_dtype(dtype)) return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent: unknown dtype %d", int(dtype));
  if (!aligned16(logits) || !aligned16(grad))
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent: logits and grad must be 16-byte aligned");
  const int vec = dtype == RF_F32 ? 4 : 8;
  if (vocab % vec != 0)
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent: vocab=%d must be a multiple of %d for %s", vocab, vec,
                dt_name(dtype));
  RF_TRY(check_dev_ptr(logits, "logits"));
  RF_TRY(check_dev_ptr(targets, "targets"));
  RF_TRY(check_dev_ptr(loss, "loss"));
  RF_TRY(check_dev_ptr(lse, "lse"));
  RF_TRY(check_dev_ptr(grad, "grad"));
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_softmax_xent: cannot resolve the device status word");
  return launched(rf::launch_xent(logits, targets, loss, lse, grad, rows, vocab, ignore_index,
                                  static_cast<rf::Dt>(dtype), st, static_cast<cudaStream_t>(stream)),
                  "rf_softmax_xent");
}

rf_status_t rf_rmsnorm_fused(const void* x, const void* residual, const void* gamma, void* out, void* residual_out,
                             int rows, int cols, float eps, rf_dtype_t dtype, void* stream) {
  if (!x || !out) return fail(RF_ERR_INVALID_ARG, "rf_rmsnorm_fused: x and out must be non-null");
  if (rows <= 0 || cols <= 0) return fail(RF_ERR_INVALID_ARG, "rf_rmsnorm_fused: sizes must be positive");
  if (!(eps >= 0.0f) || !std::isfinite(eps))
    return fail(RF_ERR_INVALID_ARG, "rf_rmsnorm_fused: eps must be finite and >= 0");
  if (!valid_dtype(dtype)) return fail(RF_ERR_INVALID_ARG, "rf_rmsnorm_fused: unknown dtype %d", int(dtype));
  if (!aligned16(x) || !aligned16(residual) || !aligned16(gamma) || !aligned16(out) || !aligned16(residual_out))
    return fail(RF_ERR_INVALID_ARG, "rf_rmsnorm_fused: pointers must be 16-byte aligned");
  const int vec = dtype == RF_F32 ? 4 : 8;
  if (cols % vec != 0)
    return fail(RF_ERR_INVALID_ARG, "rf_rmsnorm_fused: cols=%d must be a multiple of %d for %s", cols, vec,
                dt_name(dtype));
  if (cols > rf::layernorm_max_cols(static_cast<rf::Dt>(dtype)))
    return fail(RF_ERR_UNSUPPORTED, "rf_rmsnorm_fused: cols=%d exceeds %d", cols,
                rf::layernorm_max_cols(static_cast<rf::Dt>(dtype)));
  RF_TRY(check_dev_ptr(x, "x"));
  RF_TRY(check_dev_ptr(residual, "residual"));
  RF_TRY(check_dev_ptr(gamma, "gamma"));
  RF_TRY(check_dev_ptr(out, "out"));
  RF_TRY(check_dev_ptr(residual_out, "residual_out"));
  unsigned* st = rf::device_status_ptr();
  if (!st) return fail(RF_ERR_CUDA, "rf_rmsnorm_fused: cannot resolve the device status word");
  return launched(rf::launch_rmsnorm(x, residual, gamma, out, residual_out, rows, cols, eps,
                                     static_cast<rf::Dt>(dtype), st, static_cast<cudaStream_t>(stream)),
                  "rf_rmsnorm_fused");
}

size_t rf_ablation_workspace_bytes(int op, int variant, int rows, int cols, rf_dtype_t dtype) {
  if (rows <= 0 || cols <= 0 || !valid_dtype(dtype)) return static_cast<size_t>(-1);
  if (op == 0 && variant >= 0 && variant <= 3)
    return rf::ablation_ln_workspace_bytes(rows, cols, variant, static_cast<rf::Dt>(dtype));
  if (op == 1 && variant >= 0 && variant <= 2) return rf::ablation_xent_workspace_bytes(rows, variant);
  return static_cast<size_t>(-1);
}

rf_status_t rf_layernorm_ablation(const void* x, const void* residual, const void* gamma, const void* beta,
                                  void* out, int rows, int cols, float eps, int variant, void* workspace,
                                  size_t workspace_bytes, rf_dtype_t dtype, void* stream) {
  if (variant < 0 || variant > 3)
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: variant=%d must be 0..3", variant);
  if (!residual || !gamma || !beta)
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: residual, gamma and beta are required");
  if (variant == 0)
    return rf_layernorm_fused(x, residual, gamma, beta, out, nullptr, rows, cols, eps, dtype, stream);
  if (!x || !out) return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: x and out must be non-null");
  if (rows <= 0 || cols <= 0) return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: sizes must be positive");
  if (!(eps >= 0.0f) || !std::isfinite(eps))
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: eps must be finite and >= 0");
  if (!valid_dtype(dtype)) return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: unknown dtype %d", int(dtype));
  if (!aligned16(x) || !aligned16(residual) || !aligned16(gamma) || !aligned16(beta) || !aligned16(out) ||
      !aligned16(workspace))
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: pointers must be 16-byte aligned");
  const int vec = dtype == RF_F32 ? 4 : 8;
  if (cols % vec != 0)
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: cols=%d must be a multiple of %d for %s", cols, vec,
                dt_name(dtype));
  if (variant == 1 && cols > rf::kLnSmemMaxCols)
    return fail(RF_ERR_UNSUPPORTED, "rf_layernorm_ablation: cols=%d exceeds %d for the shared-memory variant",
                cols, rf::kLnSmemMaxCols);
  const size_t need = rf::ablation_ln_workspace_bytes(rows, cols, variant, static_cast<rf::Dt>(dtype));
  if (need && (!workspace || workspace_bytes < need))
    return fail(RF_ERR_INVALID_ARG, "rf_layernorm_ablation: workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : size_t(0));
  RF_TRY(check_dev_ptr(x, "x"));
  RF_TRY(check_dev_ptr(residual, "residual"));
  RF_TRY(check_dev_ptr(gamma, "gamma"));
  RF_TRY(check_dev_ptr(beta, "beta"));
  RF_TRY(check_dev_ptr(out, "out"));
  RF_TRY(check_dev_ptr(workspace, "workspace"));
  return launched(rf::launch_ln_ablation(x, residual, gamma, beta, out, rows, cols, eps, variant, workspace,
                                         static_cast<rf::Dt>(dtype), static_cast<cudaStream_t>(stream)),
                  "rf_layernorm_ablation");
}

rf_status_t rf_softmax_xent_ablation(const void* logits, const long long* targets, float* loss, float* lse,
                                     int rows, int vocab, long long ignore_index, int variant, void* workspace,
                                     size_t workspace_bytes, rf_dtype_t dtype, void* stream) {
  if (variant < 0 || variant > 2)
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent_ablation: variant=%d must be 0..2", variant);
  if (variant == 0)
    return rf_softmax_xent(logits, targets, loss, lse, nullptr, rows, vocab, ignore_index, dtype, stream);
  if (!logits || !targets || !loss)
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent_ablation: logits, targets and loss must be non-null");
  if (rows <= 0 || vocab <= 0)
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent_ablation: sizes must be positive");
  if (!valid_dtype(dtype))
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent_ablation: unknown dtype %d", int(dtype));
  if (!aligned16(logits) || !aligned16(workspace))
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent_ablation: logits and workspace must be 16-byte aligned");
  const int vec = dtype == RF_F32 ? 4 : 8;
  if (vocab % vec != 0)
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent_ablation: vocab=%d must be a multiple of %d for %s", vocab,
                vec, dt_name(dtype));
  const size_t need = rf::ablation_xent_workspace_bytes(rows, variant);
  if (need && (!workspace || workspace_bytes < need))
    return fail(RF_ERR_INVALID_ARG, "rf_softmax_xent_ablation: workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : size_t(0));
  RF_TRY(check_dev_ptr(logits, "logits"));
  RF_TRY(check_dev_ptr(targets, "targets"));
  RF_TRY(check_dev_ptr(loss, "loss"));
  RF_TRY(check_dev_ptr(lse, "lse"));
  RF_TRY(check_dev_ptr(workspace, "workspace"));
  return launched(rf::launch_xent_ablation(logits, targets, loss, lse, rows, vocab, ignore_index, variant,
                                           workspace, static_cast<rf::Dt>(dtype),
                                           static_cast<cudaStream_t>(stream)),
                  "rf_softmax_xent_ablation");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// rf_attn_decode_splitkv_noalloc: the decode entry point for callers that may
// not allocate device memory.  Its scratch (the per-split partials) lives in
// this file-scope array instead of a caller-provided workspace.  Every GPU
// that loads the library holds the array until the process exits.  Host code
// cannot use the array's name as a device address, so the address is looked
// up with cudaGetSymbolAddress once per device (on that device's first call,
// with the device current) and cached.  Nothing in the array has to start at
// zero: each call writes every partial slot before the merge reads it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_decode_scratch[RF_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

void* decode_scratch_for_current_device() {
  static std::mutex mu;
  static void* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" rf_status_t rf_attn_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                      void* o, float* lse, int B, int Hq, int Hkv, int L, int D,
                                                      int num_splits, float scale, rf_dtype_t dtype,
                                                      void* stream) {
  const size_t need = rf_attn_decode_splitkv_workspace_bytes(B, Hq, D, num_splits);
  if (need > size_t(RF_DECODE_NOALLOC_SCRATCH_BYTES))
    return fail(RF_ERR_INVALID_ARG,
                "rf_attn_decode_splitkv_noalloc: B=%d Hq=%d D=%d num_splits=%d needs %zu bytes of scratch, "
                "more than the %zu bytes built into the library; use rf_attn_decode_splitkv with a workspace",
                B, Hq, D, num_splits, need, size_t(RF_DECODE_NOALLOC_SCRATCH_BYTES));
  void* scratch = decode_scratch_for_current_device();
  if (scratch == nullptr)
    return fail(RF_ERR_CUDA, "rf_attn_decode_splitkv_noalloc: cannot resolve the scratch address on this device");
  return rf_attn_decode_splitkv(q, k_cache, v_cache, o, lse, scratch, size_t(RF_DECODE_NOALLOC_SCRATCH_BYTES), B,
                                Hq, Hkv, L, D, num_splits, scale, dtype, stream);
}
