// flamia_fwd_noalloc: the forward call for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the moment they run attention: code
// inside a custom allocator or a memory-pool callback, runtimes that hand
// kernels only pre-registered buffers, and processes whose device memory is
// fully reserved up front.  flamia_fwd needs a caller-provided workspace only
// for its device-built work list; this variant keeps that work list in a
// file-scope device array instead, so the caller passes just inputs and
// outputs.  The array is modest (kScratchBytes, about 1.6 MB) and, like any __device__
// variable, every GPU that loads the library holds it until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/flamia.h"
#include "launch.h"

namespace flamia {

int* status_word_for_current_device();  // defined in api.cu

namespace {

// Limits of the no-allocation path and the scratch they imply.
constexpr int64_t kMaxTokens = int64_t(1) << 20;   // T
constexpr int32_t kMaxDocs = 65536;                // n_docs
constexpr int32_t kMaxC = static_cast<int32_t>((kMaxTokens + kTile - 1) / kTile);
constexpr size_t kHdrBytes = 256;
constexpr size_t kDocsBytes = static_cast<size_t>(kMaxDocs) * sizeof(int32_t);
constexpr size_t kVecBytes = ((static_cast<size_t>(kMaxC) + 2) * sizeof(int32_t) + 255) / 256 * 256;
constexpr size_t kItemBytes = (static_cast<size_t>(kMaxC) + kMaxDocs) * sizeof(int4);
constexpr size_t kScratchBytes = kHdrBytes + kDocsBytes + 4 * kVecBytes + kItemBytes;   // ~1.6 MB

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct NoAllocDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  int cc_major = 0;
  int* status = nullptr;
};
NoAllocDevice g_na[kMaxDevices];
std::mutex g_na_mutex;

// One-time set-up per device, run with that device current: the host-side
// name g_noalloc_scratch is only a stand-in, so the kernels get the device
// address from cudaGetSymbolAddress.
int setup_current_device(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLAMIA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& d = g_na[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FLAMIA_ERR_LAUNCH;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FLAMIA_ERR_LAUNCH;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
      return FLAMIA_ERR_LAUNCH;
    d.status = status_word_for_current_device();
    if (!d.status) return FLAMIA_ERR_LAUNCH;
    d.scratch = static_cast<uint8_t*>(p);
    d.ready = true;
  }
  *out = &d;
  return FLAMIA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over the bf16 output O [T, Hq*d] for the forward's epilogue stores
// at d = 64: boxes of 64 columns (128 bytes, 128B swizzle) by 32 rows, one
// per softmax warp's rows.
bool o_map(CUtensorMap* m, const void* base, int64_t T, int Hq, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(Hq) * d, static_cast<cuuint64_t>(T)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(Hq) * d * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool code_map(CUtensorMap* m, const void* base, int64_t T, int H, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * d, static_cast<cuuint64_t>(T)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * d};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle sw = d == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t up256(size_t x) { return (x + 255) / 256 * 256; }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace flamia

using namespace flamia;

extern "C" int flamia_fwd_noalloc(const void* q_dev, const void* k_dev, const void* v_dev,
                                  const int32_t* cu_seqlens_dev, int32_t n_docs, int64_t T, int32_t Hq, int32_t Hkv,
                                  int32_t d, const flamia_opts* opts, void* out_dev, float* lse_dev, void* saved_dev,
                                  void* stream) {
  if (d != 64 && d != 128) return FLAMIA_ERR_UNSUPPORTED_D;
  if (T < 1 || Hq < 1 || Hkv < 1 || n_docs < 0 || Hq % Hkv != 0) return FLAMIA_ERR_ARG;
  if (T * static_cast<int64_t>(Hq > Hkv ? Hq : Hkv) * d >= (int64_t(1) << 31)) return FLAMIA_ERR_ARG;
  if (T > kMaxTokens || n_docs > kMaxDocs) return FLAMIA_ERR_NOALLOC_LIMIT;
  if (!opts || opts->c_exp < 0 || opts->tau < 0 || opts->c_exp + opts->tau > 8 ||
      (opts->causal != 0 && opts->causal != 1) || (opts->hadamard != 0 && opts->hadamard != 1) ||
      (opts->exact != 0 && opts->exact != 1) ||
      (opts->hadamard && d != 128))
    return FLAMIA_ERR_ARG;
  if (opts->nvfp4) return FLAMIA_ERR_UNSUPPORTED_OPT;   // flamia_fwd serves the NVFP4 path
  if (!q_dev || !k_dev || !v_dev || !cu_seqlens_dev || !out_dev || !lse_dev || !saved_dev) return FLAMIA_ERR_ARG;
  if (!al16(q_dev) || !al16(k_dev) || !al16(v_dev) || !al16(out_dev) || !al16(lse_dev) || !al16(saved_dev))
    return FLAMIA_ERR_ALIGN;
  NoAllocDevice* dev = nullptr;
  int rc = setup_current_device(&dev);
  if (rc != FLAMIA_OK) return rc;
  if (dev->cc_major != 10) return FLAMIA_ERR_DEVICE;

  // saved buffer: same layout as flamia_saved_bytes
  size_t o = 0;
  const size_t q_codes = o; o = up256(o + static_cast<size_t>(T) * Hq * d);
  const size_t k_codes = o; o = up256(o + static_cast<size_t>(T) * Hkv * d);
  const size_t v_codes = o; o = up256(o + static_cast<size_t>(T) * Hkv * d);
  const size_t q_scales = o; o = up256(o + static_cast<size_t>(T) * Hq);
  const size_t k_scales = o; o = up256(o + static_cast<size_t>(T) * Hkv);
  const size_t v_scales = o; o = up256(o + static_cast<size_t>(T) * Hkv);
  // exact options: V with token-block scales follows (flamia_saved_bytes_with)
  const size_t vb_codes = o; o = up256(o + static_cast<size_t>(T) * Hkv * d);
  const size_t vb_scales = o;
  uint8_t* sv = static_cast<uint8_t*>(saved_dev);

  // work list inside the static array; the plan kernel rewrites every field it
  // reads (its histograms are zeroed in the same launch), so nothing carries
  // over from the previous call
  const int cap_C = static_cast<int>((T + kTile - 1) / kTile);
  PlanView pv;
  uint8_t* base = dev->scratch;
  pv.hdr = reinterpret_cast<int32_t*>(base);
  pv.sorted_docs = reinterpret_cast<int32_t*>(base + kHdrBytes);
  pv.cnt_ge = reinterpret_cast<int32_t*>(base + kHdrBytes + kDocsBytes);
  pv.off = reinterpret_cast<int32_t*>(base + kHdrBytes + kDocsBytes + kVecBytes);
  pv.hist = reinterpret_cast<int32_t*>(base + kHdrBytes + kDocsBytes + 2 * kVecBytes);
  pv.fill = reinterpret_cast<int32_t*>(base + kHdrBytes + kDocsBytes + 3 * kVecBytes);
  pv.items = reinterpret_cast<int4*>(base + kHdrBytes + kDocsBytes + 4 * kVecBytes);
  pv.order = 0;                       // the forward's longest-first order
  pv.causal = opts->causal;
  pv.doc_first = nullptr;

  FwdArgs fa{};
  if (!code_map(&fa.tm_q, sv + q_codes, T, Hq, d) || !code_map(&fa.tm_k, sv + k_codes, T, Hkv, d) ||
      !code_map(&fa.tm_v, sv + v_codes, T, Hkv, d))
    return FLAMIA_ERR_LAUNCH;
  if (opts->exact && !code_map(&fa.tm_vb, sv + vb_codes, T, Hkv, d)) return FLAMIA_ERR_LAUNCH;
  if (d == 64 && !o_map(&fa.tm_o, out_dev, T, Hq, d)) return FLAMIA_ERR_LAUNCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_plan(cu_seqlens_dev, n_docs, T, pv, cap_C, dev->status, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  QuantLaunchArgs qa{};
  qa.t[0] = {static_cast<const __nv_bfloat16*>(q_dev), sv + q_codes, sv + q_scales, Hq, opts->hadamard, opts->exact};
  qa.t[1] = {static_cast<const __nv_bfloat16*>(k_dev), sv + k_codes, sv + k_scales, Hkv, opts->hadamard, opts->exact};
  qa.t[2] = {static_cast<const __nv_bfloat16*>(v_dev), sv + v_codes, sv + v_scales, Hkv, 0, opts->exact};
  qa.ntensors = 3;
  qa.cu = cu_seqlens_dev;
  qa.n_docs = n_docs;
  qa.T = T;
  if (launch_quantize(qa, d, false, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  if (opts->exact) {
    QuantLaunchArgs qb{};
    qb.t[0] = {static_cast<const __nv_bfloat16*>(v_dev), sv + vb_codes, sv + vb_scales, Hkv, 0, 0};
    qb.ntensors = 1;
    qb.cu = cu_seqlens_dev;
    qb.n_docs = n_docs;
    qb.T = T;
    if (launch_quantize(qb, d, false, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  }
  fa.q_scales = sv + q_scales;
  fa.vb_scales = sv + vb_scales;
  fa.k_scales = sv + k_scales;
  fa.v_scales = sv + v_scales;
  fa.cu = cu_seqlens_dev;
  fa.plan_hdr = pv.hdr;
  fa.plan_items = pv.items;
  fa.out = static_cast<__nv_bfloat16*>(out_dev);
  fa.lse = lse_dev;
  fa.status = dev->status;
  fa.T = T;
  fa.Hq = Hq;
  fa.Hkv = Hkv;
  fa.causal = opts->causal;
  fa.c_exp = opts->c_exp;
  fa.tau = static_cast<float>(opts->tau);
  fa.hadamard = opts->hadamard;
  fa.exact = opts->exact;
  fa.item_counter = pv.hdr + 6;       // zeroed by the plan kernel
  fa.schedule = opts->schedule;
  if (launch_fwd(fa, d, dev->num_sms, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  if (launch_fwd_pad(cu_seqlens_dev, n_docs, T, Hq, d, out_dev, lse_dev, dev->num_sms, st) != cudaSuccess)
    return FLAMIA_ERR_LAUNCH;
  return FLAMIA_OK;
}
