// C-ABI entry points (include/flamia.h): host-side validation, buffer layout,
// TMA tensor maps and the launch sequence of each call.  No allocation, no
// host synchronisation (except the diagnostic flamia_get_status).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/flamia.h"
#include "launch.h"

namespace flamia {
namespace {

// Device status word, one per device that loads the library.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* status = nullptr;  // device address of g_status_word
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;
thread_local int32_t t_last_launches = 0;
thread_local cudaEvent_t* t_events = nullptr;
thread_local int32_t t_nevents = 0;
// score-tile copies requested by flamia_debug_set_score_dump (s null: none)
thread_local ScoreDump t_dump_fwd{};
thread_local ScoreDump t_dump_bwd{};
// item limit of the forward's CTAs set by flamia_debug_set_item_limit (0: none)
thread_local int t_item_limit = 0;

// Record the timing event of launch slot i (if the hook is set).  Under
// stream capture it goes in as an external event record, so every replay of
// the graph records it (and it can be timed); otherwise a plain record.
inline void mark(int i, cudaStream_t st) {
  if (!t_events || i >= t_nevents) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(t_events[i], st, cudaEventRecordExternal);
  else
    cudaEventRecord(t_events[i], st);
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

// Per-device set-up on first use with that device current.
const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    d.status = static_cast<int*>(p);
    d.ready = true;
  }
  return &d;
}

constexpr size_t kAlign = 256;
// CTAs of the forward's Q/K/V quantize launch that write the rows outside
// every document (a grid-stride share each)
constexpr int kPadCtas = 16;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct SavedLayout {
  size_t q_codes, k_codes, v_codes, q_scales, k_scales, v_scales;
  size_t q4_codes = 0, k4_codes = 0, q4_scales = 0, k4_scales = 0;   // NVFP4 option
  size_t vb_codes = 0, vb_scales = 0;   // exact options: V with token-block scales
  size_t total;
  SavedLayout(int64_t T, int Hq, int Hkv, int d, bool nvfp4 = false, bool exact = false) {
    size_t o = 0;
    q_codes = o; o = align_up(o + static_cast<size_t>(T) * Hq * d);
    k_codes = o; o = align_up(o + static_cast<size_t>(T) * Hkv * d);
    v_codes = o; o = align_up(o + static_cast<size_t>(T) * Hkv * d);
    q_scales = o; o = align_up(o + static_cast<size_t>(T) * Hq);
    k_scales = o; o = align_up(o + static_cast<size_t>(T) * Hkv);
    v_scales = o; o = align_up(o + static_cast<size_t>(T) * Hkv);
    if (nvfp4) {
      q4_codes = o; o = align_up(o + static_cast<size_t>(T) * Hq * d / 2);
      k4_codes = o; o = align_up(o + static_cast<size_t>(T) * Hkv * d / 2);
      q4_scales = o; o = align_up(o + static_cast<size_t>(T) * Hq * d / 16);
      k4_scales = o; o = align_up(o + static_cast<size_t>(T) * Hkv * d / 16);
    }
    if (exact) {
      vb_codes = o; o = align_up(o + static_cast<size_t>(T) * Hkv * d);
      vb_scales = o; o = align_up(o + static_cast<size_t>(T) * Hkv);
    }
    total = o;
  }
};

struct WorkLayout {
  size_t hdr, sorted, cnt_ge, off, hist, fill, items, do_codes, do_scales, D, dqacc, doc_first, total;
  int cap_C;
  WorkLayout(int64_t T, int n_docs, int Hq, int d) {
    cap_C = static_cast<int>((T + kTile - 1) / kTile);
    const size_t cvec = static_cast<size_t>(cap_C + 2) * sizeof(int32_t);
    size_t o = 0;
    // header: plan words [0, 4), the forward's dQ-accumulator stamp (64 bit)
    // at [4, 6), the claim counter of the dynamic hand-out at 6, 7 unused
    hdr = o; o = align_up(o + 8 * sizeof(int32_t));
    sorted = o; o = align_up(o + static_cast<size_t>(n_docs > 0 ? n_docs : 1) * sizeof(int32_t));
    cnt_ge = o; o = align_up(o + cvec);
    off = o; o = align_up(o + cvec);
    hist = o; o = align_up(o + cvec);
    fill = o; o = align_up(o + cvec);
    items = o; o = align_up(o + (static_cast<size_t>(cap_C) + static_cast<size_t>(n_docs)) * sizeof(int4));
    do_codes = o; o = align_up(o + static_cast<size_t>(T) * Hq * d);
    do_scales = o; o = align_up(o + static_cast<size_t>(T) * Hq);
    D = o; o = align_up(o + static_cast<size_t>(T) * Hq * sizeof(float));
    // room for the deterministic option's 64-bit fixed-point accumulator;
    // the fp32 accumulator uses the first half
    dqacc = o; o = align_up(o + static_cast<size_t>(T) * Hq * d * sizeof(uint64_t));
    doc_first = o; o = align_up(o + static_cast<size_t>(n_docs > 0 ? n_docs : 1) * sizeof(int32_t));
    total = o;
  }
  uint64_t* dq_tag(uint8_t* base) const { return reinterpret_cast<uint64_t*>(base + hdr + 4 * sizeof(int32_t)); }
  PlanView plan(uint8_t* base) const {
    PlanView p;
    p.hdr = reinterpret_cast<int32_t*>(base + hdr);
    p.sorted_docs = reinterpret_cast<int32_t*>(base + sorted);
    p.cnt_ge = reinterpret_cast<int32_t*>(base + cnt_ge);
    p.off = reinterpret_cast<int32_t*>(base + off);
    p.hist = reinterpret_cast<int32_t*>(base + hist);
    p.fill = reinterpret_cast<int32_t*>(base + fill);
    p.items = reinterpret_cast<int4*>(base + items);
    p.order = 0;
    p.causal = 1;
    p.doc_first = reinterpret_cast<int32_t*>(base + doc_first);
    return p;
  }
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int64_t T, int Hq, int Hkv, int d, int n_docs) {
  if (d != 64 && d != 128) return FLAMIA_ERR_UNSUPPORTED_D;
  if (T < 1 || Hq < 1 || Hkv < 1 || n_docs < 0 || Hq % Hkv != 0) return FLAMIA_ERR_ARG;
  if (T * static_cast<int64_t>(Hq > Hkv ? Hq : Hkv) * d >= (int64_t(1) << 31)) return FLAMIA_ERR_ARG;
  if (T >= (int64_t(1) << 31)) return FLAMIA_ERR_ARG;
  return FLAMIA_OK;
}

int check_opts(const flamia_opts* o) {
  if (!o) return FLAMIA_ERR_ARG;
  // c + tau <= log2(448): beyond it P-hat saturates silently (Appendix B.1)
  if (o->c_exp < 0 || o->tau < 0 || o->c_exp + o->tau > 8) return FLAMIA_ERR_ARG;
  if (o->causal != 0 && o->causal != 1) return FLAMIA_ERR_ARG;
  if (o->hadamard != 0 && o->hadamard != 1) return FLAMIA_ERR_ARG;
  if (o->exact != 0 && o->exact != 1) return FLAMIA_ERR_ARG;
  if (o->schedule != 0 && o->schedule != 1) return FLAMIA_ERR_ARG;
  if (o->nvfp4 != 0 && o->nvfp4 != 1) return FLAMIA_ERR_ARG;
  if (o->nvfp4 && (o->exact || o->hadamard)) return FLAMIA_ERR_ARG;
  if (o->deterministic_dq != 0 && o->deterministic_dq != 1) return FLAMIA_ERR_ARG;
  return FLAMIA_OK;
}

// 2-D map over a [T, H*d] byte matrix of E4M3 codes, one 128-token x d box,
// swizzled to match the MMA's shared-memory layout.
bool make_code_map(CUtensorMap* m, const void* base, int64_t T, int H, int d) {
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

// The same for packed E2M1 codes [T, H*d/2] (NVFP4 option): one 128-token x
// d/2-byte box, swizzled to the 4-bit MMA's K-major layout (32B rows at
// d = 64, 64B at d = 128).
bool make_code4_map(CUtensorMap* m, const void* base, int64_t T, int H, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * d / 2, static_cast<cuuint64_t>(T)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * d / 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(d / 2), static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapSwizzle sw = d == 64 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over the fp32 dQ accumulator [T, Hq*d]: boxes of 32 floats
// (128 bytes, the widest box the 128B swizzle allows) by 128 rows for d = 128
// (one box per column strip of a CTA's tile) or by 32 rows for d = 64 (one
// box per warp's rows).
bool make_dq_map(CUtensorMap* m, const void* base, int64_t T, int Hq, int d, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(Hq) * d, static_cast<cuuint64_t>(T)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(Hq) * d * sizeof(float)};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over the bf16 output O [T, Hq*d] for the forward's epilogue stores
// at d = 64: boxes of 64 columns (128 bytes, 128B swizzle) by 32 rows, one
// per softmax warp's rows.
bool make_o_map(CUtensorMap* m, const void* base, int64_t T, int Hq, int d) {
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

const DeviceInfo* checked_device(int* err) {
  const DeviceInfo* di = device_info();
  if (!di) { *err = FLAMIA_ERR_LAUNCH; return nullptr; }
  if (di->cc_major != 10) { *err = FLAMIA_ERR_DEVICE; return nullptr; }
  *err = FLAMIA_OK;
  return di;
}

}  // namespace

// Device status word of the current device, for entry points in other files.
int* status_word_for_current_device() {
  const DeviceInfo* di = device_info();
  return di ? di->status : nullptr;
}

}  // namespace flamia

using namespace flamia;

extern "C" {

flamia_opts flamia_default_opts(void) {
  flamia_opts o;
  o.c_exp = 4;
  o.tau = 4;
  o.causal = 1;
  o.hadamard = 0;
  o.exact = 0;
  o.schedule = 0;
  o.nvfp4 = 0;
  o.deterministic_dq = 0;
  return o;
}

size_t flamia_saved_bytes(int64_t T, int32_t Hq, int32_t Hkv, int32_t d) {
  if (check_shape(T, Hq, Hkv, d, 0) != FLAMIA_OK) return 0;
  // room for every option: the NVFP4 and the exact options' pieces follow
  // the common ones at the same offset (the two are never combined)
  const size_t a = SavedLayout(T, Hq, Hkv, d, true, false).total;
  const size_t b = SavedLayout(T, Hq, Hkv, d, false, true).total;
  return a > b ? a : b;
}

size_t flamia_saved_bytes_with(int64_t T, int32_t Hq, int32_t Hkv, int32_t d, const flamia_opts* opts) {
  if (check_shape(T, Hq, Hkv, d, 0) != FLAMIA_OK || check_opts(opts) != FLAMIA_OK) return 0;
  return SavedLayout(T, Hq, Hkv, d, opts->nvfp4 != 0, opts->exact != 0).total;
}

size_t flamia_workspace_bytes(int64_t T, int32_t n_docs, int32_t Hq, int32_t Hkv, int32_t d) {
  if (check_shape(T, Hq, Hkv, d, n_docs) != FLAMIA_OK) return 0;
  return WorkLayout(T, n_docs, Hq, d).total;
}

int flamia_quantize(const void* x_dev, int64_t T, int32_t H, int32_t d, const int32_t* cu_seqlens_dev,
                    int32_t n_docs, uint8_t* codes_dev, uint8_t* scales_dev, void* stream) {
  int rc = check_shape(T, H, H, d, n_docs);
  if (rc) return rc;
  if (!x_dev || !cu_seqlens_dev || !codes_dev || !scales_dev) return FLAMIA_ERR_ARG;
  if (!aligned16(x_dev) || !aligned16(codes_dev)) return FLAMIA_ERR_ALIGN;
  const DeviceInfo* di = checked_device(&rc);
  if (!di) return rc;
  QuantLaunchArgs qa{};
  qa.t[0] = {static_cast<const __nv_bfloat16*>(x_dev), codes_dev, scales_dev, H};
  qa.ntensors = 1;
  qa.cu = cu_seqlens_dev;
  qa.n_docs = n_docs;
  qa.T = T;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_quantize(qa, d, false, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  t_last_launches = 1;
  return FLAMIA_OK;
}

int flamia_fwd(const void* q_dev, const void* k_dev, const void* v_dev, const int32_t* cu_seqlens_dev,
               int32_t n_docs, int64_t T, int32_t Hq, int32_t Hkv, int32_t d, const flamia_opts* opts,
               void* out_dev, float* lse_dev, void* saved_dev, void* work_dev, void* stream) {
  int rc = check_shape(T, Hq, Hkv, d, n_docs);
  if (rc) return rc;
  if ((rc = check_opts(opts))) return rc;
  if (opts->hadamard && d != 128) return FLAMIA_ERR_ARG;
  if (t_dump_fwd.s && (opts->exact || opts->nvfp4)) return FLAMIA_ERR_UNSUPPORTED_OPT;
  if (!q_dev || !k_dev || !v_dev || !cu_seqlens_dev || !out_dev || !lse_dev || !saved_dev || !work_dev)
    return FLAMIA_ERR_ARG;
  if (!aligned16(q_dev) || !aligned16(k_dev) || !aligned16(v_dev) || !aligned16(out_dev) || !aligned16(lse_dev) ||
      !aligned16(saved_dev) || !aligned16(work_dev))
    return FLAMIA_ERR_ALIGN;
  const DeviceInfo* di = checked_device(&rc);
  if (!di) return rc;

  const SavedLayout sl(T, Hq, Hkv, d, opts->nvfp4 != 0, opts->exact != 0);
  const WorkLayout wl(T, n_docs, Hq, d);
  uint8_t* sv = static_cast<uint8_t*>(saved_dev);
  uint8_t* wk = static_cast<uint8_t*>(work_dev);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  FwdArgs fa{};
  if (!make_code_map(&fa.tm_q, sv + sl.q_codes, T, Hq, d) || !make_code_map(&fa.tm_k, sv + sl.k_codes, T, Hkv, d) ||
      !make_code_map(&fa.tm_v, sv + sl.v_codes, T, Hkv, d))
    return FLAMIA_ERR_LAUNCH;
  if (opts->nvfp4 && (!make_code4_map(&fa.tm_q4, sv + sl.q4_codes, T, Hq, d) ||
                      !make_code4_map(&fa.tm_k4, sv + sl.k4_codes, T, Hkv, d)))
    return FLAMIA_ERR_LAUNCH;
  if (opts->exact && !make_code_map(&fa.tm_vb, sv + sl.vb_codes, T, Hkv, d)) return FLAMIA_ERR_LAUNCH;
  if (d == 64 && !make_o_map(&fa.tm_o, out_dev, T, Hq, d)) return FLAMIA_ERR_LAUNCH;

  const PlanView pv = wl.plan(wk);
  // the forward clears the backward's fp32 dQ accumulator at d = 64 (see
  // fwd.cu); at d = 128, and for the deterministic option's fixed-point
  // accumulator, the dO quantizer does it
  float* dqacc = (d == 64 && !opts->deterministic_dq) ? reinterpret_cast<float*>(wk + wl.dqacc) : nullptr;

  QuantLaunchArgs qa{};
  // side jobs in the quantize launch: the work plan, and the rows outside
  // every document with the workspace stamp
  qa.aux.n_aux = 1 + kPadCtas;
  qa.aux.pv = pv;
  qa.aux.cap_C = wl.cap_C;
  qa.aux.status = di->status;
  qa.aux.pad_out = static_cast<__nv_bfloat16*>(out_dev);
  qa.aux.pad_lse = lse_dev;
  qa.aux.pad_dqacc = dqacc;
  qa.aux.dq_tag = dqacc ? wl.dq_tag(wk) : nullptr;
  qa.aux.dq_tag_value = dq_zero_tag(T, Hq, d);
  qa.aux.Hq = Hq;
  qa.aux.d = d;
  qa.t[0] = {static_cast<const __nv_bfloat16*>(q_dev), sv + sl.q_codes, sv + sl.q_scales, Hq, opts->hadamard,
             opts->exact};
  qa.t[1] = {static_cast<const __nv_bfloat16*>(k_dev), sv + sl.k_codes, sv + sl.k_scales, Hkv, opts->hadamard,
             opts->exact};
  qa.t[2] = {static_cast<const __nv_bfloat16*>(v_dev), sv + sl.v_codes, sv + sl.v_scales, Hkv, 0, opts->exact};
  if (opts->nvfp4) {
    // the NVFP4 Q and K of the scores, next to their E4M3 codes
    qa.t[0].codes4 = sv + sl.q4_codes;
    qa.t[0].scales4 = sv + sl.q4_scales;
    qa.t[1].codes4 = sv + sl.k4_codes;
    qa.t[1].scales4 = sv + sl.k4_scales;
  }
  qa.ntensors = 3;
  qa.cu = cu_seqlens_dev;
  qa.n_docs = n_docs;
  qa.T = T;
  mark(0, st);
  if (launch_quantize(qa, d, false, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  int launches = 0;
  if (opts->exact) {
    // the exact options also keep V with token-block scales: the forward
    // folds V's per-key exponent on the diagonal tile only (FLAMIA Section
    // 3.2) and multiplies these codes on the tiles before it
    QuantLaunchArgs qb{};
    qb.t[0] = {static_cast<const __nv_bfloat16*>(v_dev), sv + sl.vb_codes, sv + sl.vb_scales, Hkv, 0, 0};
    qb.ntensors = 1;
    qb.cu = cu_seqlens_dev;
    qb.n_docs = n_docs;
    qb.T = T;
    mark(1, st);
    if (launch_quantize(qb, d, false, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
    launches = 1;
  }

  fa.q_scales = sv + sl.q_scales;
  fa.k_scales = sv + sl.k_scales;
  fa.v_scales = sv + sl.v_scales;
  fa.cu = cu_seqlens_dev;
  fa.plan_hdr = pv.hdr;
  fa.plan_items = pv.items;
  fa.out = static_cast<__nv_bfloat16*>(out_dev);
  fa.lse = lse_dev;
  fa.status = di->status;
  fa.T = T;
  fa.Hq = Hq;
  fa.Hkv = Hkv;
  fa.causal = opts->causal;
  fa.c_exp = opts->c_exp;
  fa.tau = static_cast<float>(opts->tau);
  fa.hadamard = opts->hadamard;
  fa.exact = opts->exact;
  fa.dqacc = dqacc;
  fa.dq_tag = dqacc ? wl.dq_tag(wk) : nullptr;
  fa.item_counter = pv.hdr + 6;
  fa.schedule = opts->schedule;
  fa.dump = t_dump_fwd;
  fa.debug_item_limit = t_item_limit;
  fa.nvfp4 = opts->nvfp4;
  fa.q4_scales = sv + sl.q4_scales;
  fa.k4_scales = sv + sl.k4_scales;
  fa.vb_scales = sv + sl.vb_scales;
  if (dqacc && !make_dq_map(&fa.tm_dqz, fa.dqacc, T, Hq, d, 32)) return FLAMIA_ERR_LAUNCH;
  mark(1 + launches, st);
  if (launch_fwd(fa, d, di->num_sms, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  mark(2 + launches, st);
  t_last_launches = 2 + launches;
  return FLAMIA_OK;
}

int flamia_bwd(const void* out_dev, const float* lse_dev, const void* dout_dev, const int32_t* cu_seqlens_dev,
               int32_t n_docs, int64_t T, int32_t Hq, int32_t Hkv, int32_t d, const flamia_opts* opts,
               const void* saved_dev, void* dq_dev, void* dk_dev, void* dv_dev, void* work_dev, void* stream) {
  int rc = check_shape(T, Hq, Hkv, d, n_docs);
  if (rc) return rc;
  if ((rc = check_opts(opts))) return rc;
  if (opts->hadamard && d != 128) return FLAMIA_ERR_ARG;
  if (t_dump_bwd.s && (opts->exact || opts->nvfp4 || opts->deterministic_dq)) return FLAMIA_ERR_UNSUPPORTED_OPT;
  if (!out_dev || !lse_dev || !dout_dev || !cu_seqlens_dev || !saved_dev || !dq_dev || !dk_dev || !dv_dev ||
      !work_dev)
    return FLAMIA_ERR_ARG;
  if (!aligned16(out_dev) || !aligned16(lse_dev) || !aligned16(dout_dev) || !aligned16(saved_dev) ||
      !aligned16(dq_dev) || !aligned16(dk_dev) || !aligned16(dv_dev) || !aligned16(work_dev))
    return FLAMIA_ERR_ALIGN;
  const DeviceInfo* di = checked_device(&rc);
  if (!di) return rc;

  const SavedLayout sl(T, Hq, Hkv, d, opts->nvfp4 != 0, opts->exact != 0);
  const WorkLayout wl(T, n_docs, Hq, d);
  const uint8_t* sv = static_cast<const uint8_t*>(saved_dev);
  uint8_t* wk = static_cast<uint8_t*>(work_dev);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  BwdArgs ba{};
  if (!make_code_map(&ba.tm_q, sv + sl.q_codes, T, Hq, d) || !make_code_map(&ba.tm_k, sv + sl.k_codes, T, Hkv, d) ||
      !make_code_map(&ba.tm_v, sv + sl.v_codes, T, Hkv, d) || !make_code_map(&ba.tm_do, wk + wl.do_codes, T, Hq, d) ||
      // reduce-add boxes: 32 columns x 32 rows for the d = 64 kernel, x 128
      // rows for the d = 128 one
      !make_dq_map(&ba.tm_dq, wk + wl.dqacc, T, Hq, d, d == 64 ? 32 : kTile))
    return FLAMIA_ERR_LAUNCH;
  if (opts->nvfp4 && (!make_code4_map(&ba.tm_q4, sv + sl.q4_codes, T, Hq, d) ||
                      !make_code4_map(&ba.tm_k4, sv + sl.k4_codes, T, Hkv, d)))
    return FLAMIA_ERR_LAUNCH;

  // the backward walks its key tiles document by document, so the dQ
  // partials of a document reach the fp32 accumulator while its rows are
  // in L2
  PlanView pv = wl.plan(wk);
  pv.order = 1;
  pv.causal = opts->causal;

  QuantLaunchArgs qa{};
  qa.aux.n_aux = 1;                 // the work plan rides along
  qa.aux.pv = pv;
  qa.aux.cap_C = wl.cap_C;
  qa.aux.status = di->status;
  qa.t[0] = {static_cast<const __nv_bfloat16*>(dout_dev), wk + wl.do_codes, wk + wl.do_scales, Hq, 0, opts->exact};
  qa.ntensors = 1;
  qa.cu = cu_seqlens_dev;
  qa.n_docs = n_docs;
  qa.T = T;
  qa.ex.o = static_cast<const __nv_bfloat16*>(out_dev);
  qa.ex.D = reinterpret_cast<float*>(wk + wl.D);
  qa.ex.dqacc = reinterpret_cast<float*>(wk + wl.dqacc);
  // the forward's stamp covers the fp32 accumulator only: the fixed-point
  // one is always zeroed here
  qa.ex.dq_tag = opts->deterministic_dq ? nullptr : wl.dq_tag(wk);
  qa.ex.dq_expect = dq_zero_tag(T, Hq, d);
  qa.ex.dq_fixed = opts->deterministic_dq;
  mark(0, st);
  if (launch_quantize(qa, d, true, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;

  ba.q_scales = sv + sl.q_scales;
  ba.k_scales = sv + sl.k_scales;
  ba.v_scales = sv + sl.v_scales;
  ba.do_scales = wk + wl.do_scales;
  ba.lse = lse_dev;
  ba.D = reinterpret_cast<const float*>(wk + wl.D);
  ba.cu = cu_seqlens_dev;
  ba.plan_hdr = pv.hdr;
  ba.plan_items = pv.items;
  ba.dqacc = reinterpret_cast<float*>(wk + wl.dqacc);
  ba.dk = static_cast<__nv_bfloat16*>(dk_dev);
  ba.dv = static_cast<__nv_bfloat16*>(dv_dev);
  ba.status = di->status;
  ba.T = T;
  ba.Hq = Hq;
  ba.Hkv = Hkv;
  ba.causal = opts->causal;
  ba.hadamard = opts->hadamard;
  ba.exact = opts->exact;
  ba.item_counter = pv.hdr + 6;
  ba.schedule = opts->schedule;
  ba.dump = t_dump_bwd;
  ba.nvfp4 = opts->nvfp4;
  ba.q4_scales = sv + sl.q4_scales;
  ba.k4_scales = sv + sl.k4_scales;
  ba.det_dq = opts->deterministic_dq;
  mark(1, st);
  if (launch_bwd(ba, d, di->num_sms, st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  mark(2, st);
  if (launch_bwd_finalize(cu_seqlens_dev, n_docs, T, Hq, Hkv, d, ba.dqacc, dq_dev, dk_dev, dv_dev, di->num_sms, st,
                          wl.dq_tag(wk), opts->hadamard, opts->deterministic_dq) != cudaSuccess)
    return FLAMIA_ERR_LAUNCH;
  mark(3, st);
  t_last_launches = 3;
  return FLAMIA_OK;
}

int flamia_get_status(int32_t* status_out, void* stream) {
  if (!status_out) return FLAMIA_ERR_ARG;
  const DeviceInfo* di = device_info();
  if (!di) return FLAMIA_ERR_LAUNCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  if (cudaMemcpy(&v, di->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  if (cudaMemset(di->status, 0, sizeof(int)) != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  if (cudaDeviceSynchronize() != cudaSuccess) return FLAMIA_ERR_LAUNCH;
  *status_out = v;
  return FLAMIA_OK;
}

int32_t flamia_last_launch_count(void) { return t_last_launches; }

int flamia_debug_set_score_dump(float* s_fwd_dev, float* f_fwd_dev, float* s_bwd_dev, float* f_bwd_dev, int32_t h,
                                int32_t doc, int32_t qt, int32_t kt) {
  if ((s_fwd_dev != nullptr) != (f_fwd_dev != nullptr) || (s_bwd_dev != nullptr) != (f_bwd_dev != nullptr))
    return FLAMIA_ERR_ARG;
  t_dump_fwd = ScoreDump{s_fwd_dev, f_fwd_dev, h, doc, qt, kt};
  t_dump_bwd = ScoreDump{s_bwd_dev, f_bwd_dev, h, doc, qt, kt};
  return FLAMIA_OK;
}

int flamia_debug_set_item_limit(int32_t n) {
  if (n < 0) return FLAMIA_ERR_ARG;
  t_item_limit = n;
  return FLAMIA_OK;
}

int flamia_set_launch_events(void** events, int32_t n) {
  t_events = (events && n > 0) ? reinterpret_cast<cudaEvent_t*>(events) : nullptr;
  t_nevents = t_events ? n : 0;
  return FLAMIA_OK;
}

}  // extern "C"
