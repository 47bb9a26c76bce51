// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "flamia_common.cuh"

namespace flamia {

struct QuantTensorArgs {
  const __nv_bfloat16* x;  // [T, H, d]
  uint8_t* codes;          // [T, H, d]
  uint8_t* scales;         // [H, T]
  int H;
  int rotate;              // 1: rotate each token row by H_d first (d = 128)
  int per_token;           // 1: one exponent per token row instead of per 32-token block
  uint8_t* codes4;         // NVFP4 option: E2M1 codes [T, H, d/2] (null: none)
  uint8_t* scales4;        //   and UE4M3 scales [T, H, d/16]
};

struct QuantExtraArgs {
  const __nv_bfloat16* o;  // forward output, dO mode only
  float* D;                // [H, T], dO mode only
  float* dqacc;            // [T, H, d] fp32, zeroed in dO mode unless already zero
  const uint64_t* dq_tag;  // dO mode: the workspace stamp; dqacc is zero iff
  uint64_t dq_expect;      //   *dq_tag == dq_expect (null: always zero it)
  int dq_fixed;            // 1: dqacc has 8-byte elements (deterministic option)
};

// Side jobs that ride along in the first CTAs of a quantize launch, so they
// cost no launch of their own: the work plan (one CTA) and, for the forward,
// the rows outside every document (O = 0, LSE = +inf, dQ accumulator rows 0)
// with the workspace stamp.
struct QuantAux {
  int n_aux;              // CTAs of row y = 0 taken by these jobs (0: none)
  // work plan
  PlanView pv;
  int cap_C;
  int* status;
  // padding rows (pad_out null: none)
  __nv_bfloat16* pad_out;
  float* pad_lse;
  float* pad_dqacc;       // may be null
  uint64_t* dq_tag;       // may be null: stamped with dq_tag_value
  uint64_t dq_tag_value;
  int Hq, d;
};

// The forward zeroes the fp32 dQ accumulator of the workspace it is given
// (its kernels run far below the memory bandwidth, so the writes are nearly
// free there) and stamps the workspace with this tag, derived from the shape;
// the backward's dO quantizer skips the zeroing when it finds the stamp, and
// the backward's last kernel clears the stamp (the accumulator then holds
// sums).
__host__ __device__ constexpr uint64_t dq_zero_tag(int64_t T, int Hq, int d) {
  return 0x9E3779B97F4A7C15ull ^ (static_cast<uint64_t>(T) << 24) ^ (static_cast<uint64_t>(Hq) << 8) ^
         static_cast<uint64_t>(d);
}

struct QuantLaunchArgs {
  QuantTensorArgs t[3];
  int ntensors;
  const int32_t* cu;
  int n_docs;
  int64_t T;
  QuantExtraArgs ex;
  QuantAux aux;
};

cudaError_t launch_quantize(const QuantLaunchArgs& a, int d, bool do_mode, cudaStream_t st);
// Standalone launches of the side jobs (used where no quantize launch
// precedes the attention kernel).
cudaError_t launch_plan(const int32_t* cu, int n_docs, int64_t T, const PlanView& pv, int cap_C, int* status,
                        cudaStream_t st);
// dqacc (may be null): the fp32 dQ accumulator, zeroed for rows outside the
// documents, and its stamp written once the whole accumulator is zero.
cudaError_t launch_fwd_pad(const int32_t* cu, int n_docs, int64_t T, int Hq, int d, void* out, float* lse,
                           int num_sms, cudaStream_t st, float* dqacc = nullptr, uint64_t* dq_tag = nullptr);
// dq_tag (may be null): the workspace stamp, cleared (the accumulator now holds sums).
// rotate: dQ rows are mapped back by H_d / d (Hadamard option, d = 128).
// fixed: the accumulator holds signed 64-bit sums in units of 2^-32
// (deterministic option) instead of fp32.
cudaError_t launch_bwd_finalize(const int32_t* cu, int n_docs, int64_t T, int Hq, int Hkv, int d, const void* dqacc,
                                void* dq, void* dk, void* dv, int num_sms, cudaStream_t st,
                                uint64_t* dq_tag = nullptr, int rotate = 0, int fixed = 0);

// A copy of one score tile, written only by the kernels' dump variants (a
// diagnostic that shows the backward recomputes the forward's S tile bit for
// bit): the raw fp32 accumulator of Qhat Khat^T on the codes and the factor
// 2^(E_Q(i) + E_K(g)) log2(e)/sqrt(d) each row applies to each 32-key group.
struct ScoreDump {
  float* s;   // [128 rows][128 keys]; null: no dump
  float* f;   // [128 rows][4 groups]
  int h, doc, qt, kt;   // query head, document, query tile, key tile (document-relative)
};

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;   // u8 codes [T rows][H*d cols], box d x 128
  const uint8_t* q_scales;        // [Hq, T]
  const uint8_t* k_scales;        // [Hkv, T]
  const uint8_t* v_scales;        // [Hkv, T]
  const int32_t* cu;
  const int32_t* plan_hdr;
  const int4* plan_items;
  __nv_bfloat16* out;             // [T, Hq, d]
  CUtensorMap tm_o;               // d = 64: out as [T rows][Hq*d cols] bf16, box 64 x 32 (128B swizzle)
  float* lse;                     // [Hq, T]
  int* status;
  int64_t T;
  int Hq, Hkv;
  int causal;
  int c_exp;
  float tau;
  int hadamard;                   // Q and K were rotated by H_d: scores carry 1/d
  int exact;                      // per-token Q, K, V scales; V's exponents folded into P-hat
  float* dqacc;                   // [T, Hq, d] fp32 accumulator to zero (null: none; d = 64 only)
  CUtensorMap tm_dqz;             // map over dqacc, box 32 x 32 fp32 (128B swizzle), for the zero stores
  uint64_t* dq_tag;               // the workspace stamp, withdrawn if the clearing was not completed (may be null)
  int* item_counter;              // claim counter of the dynamic hand-out (zeroed by the plan job)
  int schedule;                   // 0: dynamic hand-out, 1: static snake walk
  ScoreDump dump;                 // dump variants only
  // diagnostic (0 = off): each CTA hands out at most this many items and then
  // stops, so its other warps' waits for the next item run out and the call
  // reports a wait timeout
  int debug_item_limit;
  // exact options: V with token-block scales (codes and [Hkv, T] scale
  // bytes), multiplied on the tiles before the diagonal one
  CUtensorMap tm_vb;
  const uint8_t* vb_scales;
  // NVFP4 option: Q and K for S as E2M1 codes [T rows][H*d/2 bytes] (box
  // d/2 x 128, 32B swizzle at d = 64, 64B at d = 128) and UE4M3 scales [T, H, d/16]
  CUtensorMap tm_q4, tm_k4;
  const uint8_t* q4_scales;
  const uint8_t* k4_scales;
  int nvfp4;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  CUtensorMap tm_dq;              // fp32 dQ accumulator [T rows][Hq*d cols], box 32 x 128, 128B swizzle
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const uint8_t* do_scales;       // [Hq, T]
  const float* lse;               // [Hq, T]
  const float* D;                 // [Hq, T]
  const int32_t* cu;
  const int32_t* plan_hdr;
  const int4* plan_items;
  float* dqacc;                   // [T, Hq, d]
  __nv_bfloat16* dk;              // [T, Hkv, d]
  __nv_bfloat16* dv;              // [T, Hkv, d]
  int* status;
  int64_t T;
  int Hq, Hkv;
  int causal;
  int hadamard;                   // Q and K were rotated by H_d: scores carry 1/d, dK is mapped back
  int exact;                      // exact options: per-token operands, folded payloads (d = 64)
  int* item_counter;              // claim counter of the dynamic hand-out (zeroed by the plan job)
  int schedule;                   // 0: dynamic hand-out, 1: static snake walk
  ScoreDump dump;                 // dump variants only
  // NVFP4 option: Q and K for the recomputed S (layout as in FwdArgs)
  CUtensorMap tm_q4, tm_k4;
  const uint8_t* q4_scales;
  const uint8_t* k4_scales;
  int nvfp4;
  // deterministic option: dqacc holds signed 64-bit fixed-point sums (units
  // of 2^-32), added with integer bulk reduce-adds, one per row and 16 columns
  int det_dq;
};

// True on the first call for the current device, per call site: kernel
// attributes (the dynamic shared-memory limit) are set once per device before
// the first launch, so later launches, including ones made under stream
// capture, do nothing but launch.
inline bool first_use_on_device(std::atomic<uint64_t>& seen) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return true;
  const uint64_t bit = 1ull << dev;
  return (seen.fetch_or(bit) & bit) == 0;
}

cudaError_t launch_fwd(const FwdArgs& a, int d, int num_ctas, cudaStream_t st);
cudaError_t launch_bwd(const BwdArgs& a, int d, int num_ctas, cudaStream_t st);
cudaError_t launch_bwd_d64(const BwdArgs& a, int num_ctas, cudaStream_t st);

}  // namespace flamia
