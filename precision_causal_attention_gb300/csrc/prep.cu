// Memory-bound kernels around the attention kernels:
//   * token-block MXFP8 quantizer (Q, K, V in one launch; dO with D and the
//     dQ-accumulator initialisation in another),
//   * device work-list builder (longest-first schedule),
//   * padding-row writer (forward) and dQ finalisation (backward).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "flamia_common.cuh"
#include "launch.h"

namespace flamia {

// ============================================================== quantizer
// One warp per (32-token chunk [32c, 32c+32), head): it quantizes every
// document-local 32-token block whose first token lies in that chunk, so each
// block is handled by exactly one warp and no block crosses a document
// boundary (FLAMIA Sections 3.1, 3.6.1).  A block is <= 32 tokens x d
// channels: the warp holds it in registers, takes the maximum magnitude with
// one warp reduction, derives the round-up exponent (Section 3.2) and writes
// the E4M3 codes plus one scale byte per token.
//
// dO mode additionally computes D_t = sum_c dOhat_tc O_tc from the codes it
// just wrote (Section 3.3: D from the same quantized dO that dP uses) and
// zeroes the fp32 dQ accumulator rows of its chunk (Section 3.5.1: the dO
// launch initialises the dQ accumulator).

template <int D>
struct QuantGeom {
  static constexpr int kLanesPerRow = D * 2 / 16;     // 16-byte pieces per token row
  static constexpr int kRowsPerPass = 32 / kLanesPerRow;
  static constexpr int kPasses = kBlock / kRowsPerPass;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hh);
}

template <int D, bool kDoMode, bool kPerToken>
__device__ __forceinline__ void quantize_block(const QuantTensorArgs& ta, const QuantExtraArgs& ex, int64_t T, int H,
                                               int h, int64_t b0, int nrows, int lane) {
  using G = QuantGeom<D>;
  const int sub = lane % G::kLanesPerRow;
  const int rsub = lane / G::kLanesPerRow;
  const int col = sub * 8;
  const int64_t row_stride = static_cast<int64_t>(H) * D;
  const __nv_bfloat16* xb = ta.x + (b0 * H + h) * D + col;
  uint4 v[G::kPasses];
  // dO mode: the O rows the D sums need, loaded before any store so that they
  // are in flight together with the dO rows (a load issued after a store to
  // the code array could not be moved above it)
  uint4 ov[kDoMode ? G::kPasses : 1];
  if constexpr (kDoMode) {
#pragma unroll
    for (int p = 0; p < G::kPasses; ++p) {
      const int r = p * G::kRowsPerPass + rsub;
      ov[p] = r < nrows ? __ldg(reinterpret_cast<const uint4*>(ex.o + (b0 * H + h) * D + col + r * row_stride))
                        : make_uint4(0, 0, 0, 0);
    }
  }
  // Hadamard option (d = 128): every token row is rotated by H_128 in fp32
  // and the rotated values are coded; the rotation is recomputed in the
  // coding pass rather than kept (it is cheap next to the loads)
  const bool rot = (D == 128) && ta.rotate;
  auto row_values = [&](const uint4& q, float (&x)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = bf16_lo(w[j]);
      x[2 * j + 1] = bf16_hi(w[j]);
    }
    if (rot) fwht128_row(x, sub);
  };
#pragma unroll
  for (int p = 0; p < G::kPasses; ++p) {
    const int r = p * G::kRowsPerPass + rsub;
    if (r < nrows) {
      v[p] = __ldg(reinterpret_cast<const uint4*>(xb + r * row_stride));
    } else {
      v[p] = make_uint4(0, 0, 0, 0);
    }
  }
  // exponent of the block (token blocks) or of each pass's row (per-token
  // scales of the exact options, Appendix A.3)
  int Eb = 0;
  float inv_b = 1.f;
  int Ep[kPerToken ? G::kPasses : 1];
  if constexpr (kPerToken) {
#pragma unroll
    for (int p = 0; p < G::kPasses; ++p) {
      uint32_t b;
      if (!rot) {
        // bf16 magnitudes order like their 15-bit patterns (see below)
        uint32_t m2 = __vmaxu2(__vmaxu2(v[p].x & 0x7FFF7FFFu, v[p].y & 0x7FFF7FFFu),
                               __vmaxu2(v[p].z & 0x7FFF7FFFu, v[p].w & 0x7FFF7FFFu));
        b = max(m2 & 0xFFFFu, m2 >> 16) << 16;
      } else {
        float x[8];
        row_values(v[p], x);
        float am = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(x[j]));
        b = __float_as_uint(am);
      }
#pragma unroll
      for (int m = G::kLanesPerRow / 2; m >= 1; m >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, m));
      Ep[p] = roundup_exponent_from_bits(b);
    }
  } else {
    float amax = 0.f;
    if (!rot) {
      // bf16 magnitudes order like their 15-bit patterns: the block maximum
      // comes from packed integer maxima, without converting to fp32 here
      uint32_t m2 = 0;
#pragma unroll
      for (int p = 0; p < G::kPasses; ++p) {
        m2 = __vmaxu2(m2, v[p].x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[p].y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[p].z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[p].w & 0x7FFF7FFFu);
      }
      amax = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
    } else {
#pragma unroll
      for (int p = 0; p < G::kPasses; ++p) {
        float x[8];
        row_values(v[p], x);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
      }
    }
    const uint32_t abits = warp_max_u32(__float_as_uint(amax));
    Eb = roundup_exponent_from_bits(abits);
    // E <= 120 for any finite bf16 input (127 rotated), so 2^-E is a normal fp32 number.
    inv_b = pow2f(-(Eb > 126 ? 126 : Eb));
  }
  uint8_t* cb = ta.codes + (b0 * H + h) * D + col;
#pragma unroll
  for (int p = 0; p < G::kPasses; ++p) {
    const int r = p * G::kRowsPerPass + rsub;
    const int E = kPerToken ? Ep[p] : Eb;
    const float inv_scale = kPerToken ? pow2f(-(E > 126 ? 126 : E)) : inv_b;
    float x[8];
    row_values(v[p], x);
    uint16_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // x * 2^-E is exact (power-of-two scaling); the convert rounds once.
      c[j] = cvt_e4m3x2(__fmul_rn(x[2 * j], inv_scale), __fmul_rn(x[2 * j + 1], inv_scale));
    }
    float dsum = 0.f;
    if (r < nrows) {
      uint2 packed;
      packed.x = static_cast<uint32_t>(c[0]) | (static_cast<uint32_t>(c[1]) << 16);
      packed.y = static_cast<uint32_t>(c[2]) | (static_cast<uint32_t>(c[3]) << 16);
      *reinterpret_cast<uint2*>(cb + r * row_stride) = packed;
      if constexpr (kDoMode) {
        const uint32_t ow[4] = {ov[p].x, ov[p].y, ov[p].z, ov[p].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 dv = e4m3x2_to_float2(c[j]);
          dsum = fmaf(dv.x, bf16_lo(ow[j]), dsum);
          dsum = fmaf(dv.y, bf16_hi(ow[j]), dsum);
        }
      }
    }
    if constexpr (kDoMode) {
      // reduce over the lanes that share this token row
#pragma unroll
      for (int m = G::kLanesPerRow / 2; m >= 1; m >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, m);
      if (sub == 0 && r < nrows) {
        // D = 2^E * sum(code values * O); the power-of-two factor is exact
        ex.D[static_cast<int64_t>(h) * T + b0 + r] = ldexpf(dsum, E);
      }
    }
    if (kPerToken && sub == 0 && r < nrows) ta.scales[static_cast<int64_t>(h) * T + b0 + r] = static_cast<uint8_t>(E + 127);
  }
  if (!kPerToken && lane < nrows) ta.scales[static_cast<int64_t>(h) * T + b0 + lane] = static_cast<uint8_t>(Eb + 127);
}

// ---------------------------------------------------------------- NVFP4
// The mixed NVFP4/FP8 path (FLAMIA Section 3.4): Q and K for the scores as
// E2M1 codes with one UE4M3 scale per 16 head-dimension elements of each
// token.  The scale is the smallest UE4M3 value s with 6 s >= the group's
// largest magnitude (6 s is exact in fp32, so the comparison is exact), and
// an element's code is E2M1 round-to-nearest-even of the fp32 quotient x / s.
__device__ __forceinline__ uint8_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}" : "=h"(r) : "f"(hi), "f"(lo));
  return static_cast<uint8_t>(r);
}
// value of a UE4M3 byte b in 0..0x7E
__device__ __forceinline__ float ue4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xF, m = b & 7;
  return e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}
// smallest UE4M3 byte c with 6 value(c) >= amax (0 for amax = 0, 0x7E at most):
// the nearest byte to amax / 6, then one step up or down where it misses
__device__ __forceinline__ uint32_t ue4m3_roundup(float amax) {
  if (!(amax > 0.f)) return 0u;
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(amax / 6.f));
  uint32_t c = r & 0x7Fu;
  if (c == 0) c = 1;
  if (c < 0x7E && 6.f * ue4m3_value(c) < amax) ++c;
  if (c > 1 && 6.f * ue4m3_value(c - 1) >= amax) --c;
  return c;
}

// NVFP4 codes of the tokens [t0, t1) of head h; tokens outside [lo, hi) (no
// document) get codes 0 and scales 0.  8 lanes per token row and 16-element
// group pairs at d = 64, 16 lanes at d = 128.  Every lane of the warp calls it.
template <int D>
__device__ void nvfp4_chunk(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                            int H, int h, int64_t t0, int64_t t1, int64_t lo, int64_t hi, int lane) {
  constexpr int kLanesPerRow = D / 8, kRowsPerPass = 32 / kLanesPerRow, kPasses = kBlock / kRowsPerPass;
  const int sub = lane % kLanesPerRow, rsub = lane / kLanesPerRow;
  // every row of the chunk is loaded before any is coded, so the loads are
  // in flight together
  uint4 vr[kPasses];
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int64_t t = t0 + p * kRowsPerPass + rsub;
    const bool in = t < t1 && t >= lo && t < hi;
    vr[p] = in ? __ldg(reinterpret_cast<const uint4*>(x + (t * H + h) * D + sub * 8)) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int64_t t = t0 + p * kRowsPerPass + rsub;
    const uint4 v = vr[p];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    float am = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(f[j]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));   // the group's other 8 elements
    const uint32_t sc = ue4m3_roundup(am);
    const float s = ue4m3_value(sc);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float q0 = sc ? __fdiv_rn(f[2 * j], s) : 0.f, q1 = sc ? __fdiv_rn(f[2 * j + 1], s) : 0.f;
      packed |= static_cast<uint32_t>(cvt_e2m1x2(q0, q1)) << (8 * j);
    }
    if (t < t1) {
      reinterpret_cast<uint32_t*>(codes + (t * H + h) * (D / 2))[sub] = packed;
      if ((sub & 1) == 0) scales[(t * H + h) * (D / 16) + sub / 2] = static_cast<uint8_t>(sc);
    }
  }
}

// side jobs of a quantize launch (defined with their standalone kernels below)
__device__ __noinline__ void plan_body(const int32_t* __restrict__ cu, int n_docs, int64_t T, PlanView pv, int cap_C,
                                       int* status);
__device__ __noinline__ void pad_body(const int32_t* __restrict__ cu, int n_docs, int64_t T, int Hq, int d,
                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                      float* __restrict__ dqacc, uint64_t* dq_tag, uint64_t dq_tag_value, int cta,
                                      int ncta);

template <int D, bool kDoMode, bool kPerToken>
__global__ void __launch_bounds__(256, D == 64 ? (kDoMode ? 2 : 3) : (kDoMode || kPerToken ? 1 : 2)) quantize_kernel(const __grid_constant__ QuantLaunchArgs args) {
  const int lane = threadIdx.x & 31;
  const int tsel = blockIdx.y;
  int bx = static_cast<int>(blockIdx.x);
  if (tsel == 0 && args.aux.n_aux > 0) {
    // the first CTAs, scheduled first, run the side jobs
    if (bx == 0) {
      if (args.aux.pv.hdr) plan_body(args.cu, args.n_docs, args.T, args.aux.pv, args.aux.cap_C, args.aux.status);
      return;
    }
    if (bx < args.aux.n_aux) {
      if (args.aux.pad_out)
        pad_body(args.cu, args.n_docs, args.T, args.aux.Hq, args.aux.d, args.aux.pad_out, args.aux.pad_lse,
                 args.aux.pad_dqacc, args.aux.dq_tag, args.aux.dq_tag_value, bx - 1, args.aux.n_aux - 1);
      return;
    }
    bx -= args.aux.n_aux;
  }
  const QuantTensorArgs& ta = args.t[tsel];
  const int H = ta.H;
  const int64_t T = args.T;
  const int64_t nchunks = (T + kBlock - 1) / kBlock;
  const int64_t wid = static_cast<int64_t>(bx) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (wid >= nchunks * H) return;
  const int64_t chunk = wid / H;
  const int h = static_cast<int>(wid % H);
  const int64_t t0 = chunk * kBlock;
  const int64_t t1 = (t0 + kBlock < T) ? t0 + kBlock : T;

  if (kDoMode && (args.ex.dq_tag == nullptr || *args.ex.dq_tag != args.ex.dq_expect)) {
    // zero the dQ accumulator rows of this chunk and head (unless the
    // forward left it zero): D fp32 elements per row, or D 64-bit integers
    // with the deterministic option
    uint4* acc = reinterpret_cast<uint4*>(args.ex.dqacc);
    const int per_row = args.ex.dq_fixed ? D / 2 : D / 4;
    for (int i = lane; i < static_cast<int>(t1 - t0) * per_row; i += 32) {
      const int64_t t = t0 + i / per_row;
      acc[(t * H + h) * per_row + (i % per_row)] = make_uint4(0, 0, 0, 0);
    }
  }
  const int n_docs = args.n_docs;
  const int32_t* cu = args.cu;
  {
    // Tokens outside every document get code 0 and scale byte 0, so the MMAs
    // that read them inside a partial tile multiply exact zeros by finite codes.
    int64_t lo = n_docs > 0 ? __ldg(cu) : T;
    int64_t hi = n_docs > 0 ? __ldg(cu + n_docs) : T;
    lo = lo < 0 ? 0 : (lo > T ? T : lo);
    hi = hi < lo ? lo : (hi > T ? T : hi);
    if (t0 < lo || t1 > hi) {
      constexpr int pieces = D / 16;
      const int64_t row_stride = static_cast<int64_t>(H) * D;
      for (int i = lane; i < kBlock * pieces; i += 32) {
        const int64_t t = t0 + i / pieces;
        if (t < t1 && (t < lo || t >= hi))
          reinterpret_cast<uint4*>(ta.codes + t * row_stride + static_cast<int64_t>(h) * D)[i % pieces] =
              make_uint4(0, 0, 0, 0);
      }
      const int64_t t = t0 + lane;
      if (t < t1 && (t < lo || t >= hi)) ta.scales[static_cast<int64_t>(h) * T + t] = 0;
    }
  }
  if (ta.codes4 != nullptr) {
    int64_t lo = n_docs > 0 ? __ldg(cu) : T;
    int64_t hi = n_docs > 0 ? __ldg(cu + n_docs) : T;
    lo = lo < 0 ? 0 : (lo > T ? T : lo);
    hi = hi < lo ? lo : (hi > T ? T : hi);
    nvfp4_chunk<D>(ta.x, ta.codes4, ta.scales4, H, h, t0, t1, lo, hi, lane);
  }
  if (n_docs <= 0) return;
  int r = find_doc(cu, n_docs, t0);
  for (; r < n_docs; ++r) {
    int64_t s = __ldg(cu + r), e = __ldg(cu + r + 1);
    if (s >= t1) break;
    // tolerate malformed tables: never touch tokens outside [0, T)
    s = s < 0 ? 0 : s;
    e = e > T ? T : e;
    if (e <= s || e <= t0) continue;
    const int64_t bs = (t0 <= s) ? s : s + ((t0 - s + kBlock - 1) / kBlock) * kBlock;
    if (bs < e && bs < t1) {
      const int64_t be = (bs + kBlock < e) ? bs + kBlock : e;
      quantize_block<D, kDoMode, kPerToken>(ta, args.ex, T, H, h, bs, static_cast<int>(be - bs), lane);
    }
  }
}

cudaError_t launch_quantize(const QuantLaunchArgs& a, int d, bool do_mode, cudaStream_t st) {
  int hmax = 0;
  for (int i = 0; i < a.ntensors; ++i) hmax = a.t[i].H > hmax ? a.t[i].H : hmax;
  const int64_t nchunks = (a.T + kBlock - 1) / kBlock;
  const int64_t warps = nchunks * hmax;
  dim3 grid(static_cast<unsigned>((warps + 7) / 8 + a.aux.n_aux), a.ntensors);
  // per-token scales: every tensor of a launch uses the same mode (exact
  // options)
  const bool per_token = a.t[0].per_token != 0;
  for (int i = 1; i < a.ntensors; ++i)
    if ((a.t[i].per_token != 0) != per_token) return cudaErrorInvalidValue;
  if (d == 64) {
    if (do_mode) {
      if (per_token) quantize_kernel<64, true, true><<<grid, 256, 0, st>>>(a);
      else quantize_kernel<64, true, false><<<grid, 256, 0, st>>>(a);
    } else if (per_token) quantize_kernel<64, false, true><<<grid, 256, 0, st>>>(a);
    else quantize_kernel<64, false, false><<<grid, 256, 0, st>>>(a);
  } else {
    if (do_mode) {
      if (per_token) quantize_kernel<128, true, true><<<grid, 256, 0, st>>>(a);
      else quantize_kernel<128, true, false><<<grid, 256, 0, st>>>(a);
    } else if (per_token) quantize_kernel<128, false, true><<<grid, 256, 0, st>>>(a);
    else quantize_kernel<128, false, false><<<grid, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

// ============================================================== work plan
// One CTA validates cu_seqlens and builds the longest-first schedule of
// FLAMIA Section 3.6.2 on the device (no host synchronisation): a counting
// sort of the documents by their tile count nt, plus the bucket offsets from
// which every kernel decodes item u -> (document, cost).  Runs on any block
// size (loops stride by blockDim.x); every thread of the block must call it.
__device__ __noinline__ void plan_body(const int32_t* __restrict__ cu, int n_docs, int64_t T, PlanView pv, int cap_C,
                                       int* status) {
  __shared__ int s_bad;
  __shared__ int s_max;
  if (threadIdx.x == 0) {
    s_bad = 0;
    s_max = 0;
  }
  __syncthreads();
  int bad = 0, mx = 0;
  for (int r = threadIdx.x; r < n_docs; r += blockDim.x) {
    const int64_t s = cu[r], e = cu[r + 1];
    if (s < 0 || e < s || e > T) {
      bad = 1;
    } else {
      const int nt = static_cast<int>((e - s + kTile - 1) / kTile);
      mx = nt > mx ? nt : mx;
    }
  }
  if (bad) atomicOr(&s_bad, 1);
  atomicMax(&s_max, mx);
  __syncthreads();
  const int C = s_max;
  if (s_bad || C > cap_C) {
    if (threadIdx.x == 0) {
      report_status(status, kStatusBadSeqlens);
      pv.hdr[0] = 0; pv.hdr[1] = 0; pv.hdr[2] = 0; pv.hdr[3] = n_docs;
      pv.hdr[6] = 0;
    }
    return;
  }
  for (int c = threadIdx.x; c < C + 2; c += blockDim.x) { pv.hist[c] = 0; pv.fill[c] = 0; }
  __syncthreads();
  for (int r = threadIdx.x; r < n_docs; r += blockDim.x) {
    const int nt = static_cast<int>((cu[r + 1] - cu[r] + kTile - 1) / kTile);
    if (nt > 0) atomicAdd(&pv.hist[nt], 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    pv.cnt_ge[C + 1] = 0;
    pv.off[C + 1] = 0;
    pv.cnt_ge[0] = 0;
    int run = 0;
    for (int c = C; c >= 1; --c) { run += pv.hist[c]; pv.cnt_ge[c] = run; }
    int o = 0;
    for (int c = C; c >= 1; --c) { pv.off[c] = o; o += pv.cnt_ge[c]; }
    pv.off[0] = o;
    pv.hdr[0] = o;          // items per head = sum of nt
    pv.hdr[1] = C;
    pv.hdr[2] = 1;
    pv.hdr[3] = n_docs;
    pv.hdr[6] = 0;          // claim counter of the dynamic hand-out
  }
  __syncthreads();
  for (int r = threadIdx.x; r < n_docs; r += blockDim.x) {
    const int nt = static_cast<int>((cu[r + 1] - cu[r] + kTile - 1) / kTile);
    if (nt > 0) {
      const int pos = pv.cnt_ge[nt + 1] + atomicAdd(&pv.fill[nt], 1);
      pv.sorted_docs[pos] = r;
    }
  }
  __syncthreads();
  const int n_items = pv.hdr[0];
  if (pv.order == 1) {
    // document-major records: an exclusive scan of nt over the sorted
    // documents (each thread a contiguous chunk, then a block scan of the
    // chunk sums) gives each document's first item; item u then belongs to
    // the last document whose first item is <= u
    __shared__ int s_part[1024];
    const int n_sorted = pv.cnt_ge[1];
    const int per = (n_sorted + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
    const int lo = min(static_cast<int>(threadIdx.x) * per, n_sorted), hi = min(lo + per, n_sorted);
    int local = 0;
    for (int p = lo; p < hi; ++p) {
      const int r = pv.sorted_docs[p];
      local += static_cast<int>((cu[r + 1] - cu[r] + kTile - 1) / kTile);
    }
    s_part[threadIdx.x] = local;
    __syncthreads();
    for (int off = 1; off < static_cast<int>(blockDim.x); off <<= 1) {
      const int v = static_cast<int>(threadIdx.x) >= off ? s_part[threadIdx.x - off] : 0;
      __syncthreads();
      s_part[threadIdx.x] += v;
      __syncthreads();
    }
    int run = s_part[threadIdx.x] - local;
    for (int p = lo; p < hi; ++p) {
      pv.doc_first[p] = run;
      const int r = pv.sorted_docs[p];
      run += static_cast<int>((cu[r + 1] - cu[r] + kTile - 1) / kTile);
    }
    __syncthreads();
    for (int u = threadIdx.x; u < n_items; u += blockDim.x) {
      int a = 0, b = n_sorted - 1;      // largest p with doc_first[p] <= u
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (pv.doc_first[mid] <= u) a = mid; else b = mid - 1;
      }
      const int doc = pv.sorted_docs[a];
      const int s0 = cu[doc];
      const int L = cu[doc + 1] - s0;
      const int nt = (L + kTile - 1) / kTile;
      const int kt = u - pv.doc_first[a];
      // the backward decodes a causal item's key tile as nt - c, a
      // non-causal one's as c - 1
      pv.items[u] = make_int4(doc, pv.causal ? nt - kt : kt + 1, s0, L);
    }
    return;
  }
  // one record per item, so the attention kernels decode an item with one load
  for (int u = threadIdx.x; u < n_items; u += blockDim.x) {
    int lo = 1, hi = C;                 // smallest c with off[c] <= u
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pv.off[mid] <= u) hi = mid; else lo = mid + 1;
    }
    const int doc = pv.sorted_docs[u - pv.off[lo]];
    const int s0 = cu[doc];
    pv.items[u] = make_int4(doc, lo, s0, cu[doc + 1] - s0);
  }
}

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ cu, int n_docs, int64_t T,
                                                    PlanView pv, int cap_C, int* status) {
  plan_body(cu, n_docs, T, pv, cap_C, status);
}

cudaError_t launch_plan(const int32_t* cu, int n_docs, int64_t T, const PlanView& pv, int cap_C, int* status,
                        cudaStream_t st) {
  plan_kernel<<<1, 1024, 0, st>>>(cu, n_docs, T, pv, cap_C, status);
  return cudaGetLastError();
}

// ============================================================== padding rows / dQ finalisation
// Token range [lo, hi) covered by documents, clamped to [0, T].
__device__ __forceinline__ void doc_span(const int32_t* cu, int n_docs, int64_t T, int64_t& lo, int64_t& hi) {
  const int64_t first = n_docs > 0 ? cu[0] : T;
  const int64_t last = n_docs > 0 ? cu[n_docs] : T;
  lo = first < 0 ? 0 : (first > T ? T : first);
  hi = last < lo ? lo : (last > T ? T : last);
}

// Rows outside every document: O = 0, LSE = +inf (FLAMIA Section 3.6.1), and
// the same rows of the fp32 dQ accumulator zeroed.  Block `cta` of `ncta`
// takes a grid-stride share.  The attention kernels never write these rows,
// so this may run before or after them; the stamp says the accumulator is
// zero once the forward kernel (which zeroes the rows inside the documents)
// has run too.
__device__ __noinline__ void pad_body(const int32_t* __restrict__ cu, int n_docs, int64_t T, int Hq, int d,
                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                      float* __restrict__ dqacc, uint64_t* dq_tag, uint64_t dq_tag_value, int cta,
                                      int ncta) {
  int64_t lo, hi;
  doc_span(cu, n_docs, T, lo, hi);
  const int64_t npad = lo + (T - hi);
  const int64_t per_tok = static_cast<int64_t>(Hq) * d / 8;
  const int64_t stride = static_cast<int64_t>(ncta) * blockDim.x;
  for (int64_t i = cta * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < npad * per_tok; i += stride) {
    const int64_t k = i / per_tok;
    const int64_t t = k < lo ? k : hi + (k - lo);
    reinterpret_cast<uint4*>(out)[t * per_tok + (i % per_tok)] = make_uint4(0, 0, 0, 0);
    if (dqacc) {   // the same rows of the fp32 accumulator: 2 x 16 bytes per 8 elements
      reinterpret_cast<uint4*>(dqacc)[(t * per_tok + (i % per_tok)) * 2] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(dqacc)[(t * per_tok + (i % per_tok)) * 2 + 1] = make_uint4(0, 0, 0, 0);
    }
  }
  if (dq_tag && cta == 0 && threadIdx.x == 0) *dq_tag = dq_tag_value;
  for (int64_t i = cta * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < npad * Hq; i += stride) {
    const int64_t k = i / Hq;
    const int64_t t = k < lo ? k : hi + (k - lo);
    lse[(i % Hq) * T + t] = __int_as_float(0x7f800000);
  }
}

__global__ void fwd_pad_kernel(const int32_t* __restrict__ cu, int n_docs, int64_t T, int Hq, int d,
                               __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* __restrict__ dqacc,
                               uint64_t* dq_tag) {
  pad_body(cu, n_docs, T, Hq, d, out, lse, dqacc, dq_tag, dq_zero_tag(T, Hq, d), blockIdx.x, gridDim.x);
}

cudaError_t launch_fwd_pad(const int32_t* cu, int n_docs, int64_t T, int Hq, int d, void* out, float* lse,
                           int num_sms, cudaStream_t st, float* dqacc, uint64_t* dq_tag) {
  fwd_pad_kernel<<<num_sms, 256, 0, st>>>(cu, n_docs, T, Hq, d, static_cast<__nv_bfloat16*>(out), lse, dqacc, dq_tag);
  return cudaGetLastError();
}

// dq = bf16(acc / sqrt(d)) for every row; dk = dv = 0 on rows outside every document.
// kFixed: the accumulator holds signed 64-bit sums in units of 2^-32
// (deterministic option), converted with one rounding to fp32.
template <bool kFixed>
__global__ void bwd_finalize_kernel(const int32_t* __restrict__ cu, int n_docs, int64_t T, int Hq, int Hkv, int d,
                                    const void* __restrict__ dqacc, __nv_bfloat16* __restrict__ dq,
                                    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                                    uint64_t* dq_tag, int convert_dq) {
  if (dq_tag && blockIdx.x == 0 && threadIdx.x == 0) *dq_tag = 0;   // the accumulator holds sums now
  const float scale = d == 64 ? 0.125f : 0.08838834764831845f;  // 1/sqrt(d)
  const int64_t n4 = T * Hq * d / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // four independent 16-byte (fixed point: 32-byte) loads in flight per thread
  constexpr int kU = 4;
  auto convert = [&](int64_t i, float4 a) {
    __nv_bfloat162 lo2 = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    __nv_bfloat162 hi2 = __floats2bfloat162_rn(a.z * scale, a.w * scale);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo2);
    o.y = *reinterpret_cast<uint32_t*>(&hi2);
    reinterpret_cast<uint2*>(dq)[i] = o;
  };
  auto load = [&](int64_t i) -> float4 {
    if constexpr (kFixed) {
      constexpr float kUnit = 2.3283064365386963e-10f;   // 2^-32
      const longlong2* p = reinterpret_cast<const longlong2*>(dqacc) + 2 * i;
      const longlong2 a = __ldcs(p), b = __ldcs(p + 1);
      return make_float4(__ll2float_rn(a.x) * kUnit, __ll2float_rn(a.y) * kUnit, __ll2float_rn(b.x) * kUnit,
                         __ll2float_rn(b.y) * kUnit);
    } else {
      return __ldcs(reinterpret_cast<const float4*>(dqacc) + i);
    }
  };
  int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (!convert_dq) i = n4;
  for (; i + (kU - 1) * stride < n4; i += kU * stride) {
    float4 a[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) a[u] = load(i + u * stride);
#pragma unroll
    for (int u = 0; u < kU; ++u) convert(i + u * stride, a[u]);
  }
  for (; i < n4; i += stride) convert(i, load(i));
  int64_t lo, hi;
  doc_span(cu, n_docs, T, lo, hi);
  const int64_t npad = lo + (T - hi);
  const int64_t per_tok = static_cast<int64_t>(Hkv) * d / 8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < npad * per_tok; i += stride) {
    const int64_t k = i / per_tok;
    const int64_t t = k < lo ? k : hi + (k - lo);
    reinterpret_cast<uint4*>(dk)[t * per_tok + (i % per_tok)] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(dv)[t * per_tok + (i % per_tok)] = make_uint4(0, 0, 0, 0);
  }
}

// Hadamard option (d = 128): dQ of the rotated Q mapped back, dq = bf16(acc H_128
// / 128 / sqrt(d)); a half-warp per row (8 columns per lane), rows grid-strided.
template <bool kFixed>
__global__ void bwd_finalize_rot_kernel(int64_t rows, const void* __restrict__ dqacc,
                                        __nv_bfloat16* __restrict__ dq) {
  const int lane = threadIdx.x & 31, sub = lane & 15;
  const int64_t half = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int64_t nhalf = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 4;
  const float scale = 0.08838834764831845f / 128.f;    // 1/sqrt(128) and 1/128
  // the loop count is the same for both half-warps of a warp (the shuffles
  // need every lane): rows past the end are computed on zeros and not stored
  const int64_t iters = (rows + nhalf - 1) / nhalf;
  for (int64_t k = 0; k < iters; ++k) {
    const int64_t r = half + k * nhalf;
    float x[8];
    if (r < rows) {
      if constexpr (kFixed) {
        constexpr float kUnit = 2.3283064365386963e-10f;   // 2^-32
        const longlong2* p = reinterpret_cast<const longlong2*>(dqacc) + (r * 128 + 8 * sub) / 2;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const longlong2 a = __ldcs(p + j);
          x[2 * j] = __ll2float_rn(a.x) * kUnit;
          x[2 * j + 1] = __ll2float_rn(a.y) * kUnit;
        }
      } else {
        const float* f = static_cast<const float*>(dqacc);
        const float4 a0 = __ldcs(reinterpret_cast<const float4*>(f + r * 128 + 8 * sub));
        const float4 a1 = __ldcs(reinterpret_cast<const float4*>(f + r * 128 + 8 * sub + 4));
        x[0] = a0.x; x[1] = a0.y; x[2] = a0.z; x[3] = a0.w; x[4] = a1.x; x[5] = a1.y; x[6] = a1.z; x[7] = a1.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = 0.f;
    }
    fwht128_row(x, sub);
    if (r < rows) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * j] * scale, x[2 * j + 1] * scale);
        w[j] = *reinterpret_cast<uint32_t*>(&p);
      }
      *reinterpret_cast<uint4*>(dq + r * 128 + 8 * sub) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <bool kFixed>
static void launch_finalize_t(const int32_t* cu, int n_docs, int64_t T, int Hq, int Hkv, int d, const void* dqacc,
                              void* dq, void* dk, void* dv, int num_sms, cudaStream_t st, uint64_t* dq_tag,
                              int rotate) {
  const bool rot = rotate && d == 128;
  // with the rotation, the plain kernel zeroes dK, dV outside the documents
  // and clears the stamp; the rotated dQ comes from the row-wise kernel
  bwd_finalize_kernel<kFixed><<<num_sms * 4, 256, 0, st>>>(cu, n_docs, T, Hq, Hkv, d, dqacc,
                                                           static_cast<__nv_bfloat16*>(dq),
                                                           static_cast<__nv_bfloat16*>(dk),
                                                           static_cast<__nv_bfloat16*>(dv), dq_tag, rot ? 0 : 1);
  if (rot) bwd_finalize_rot_kernel<kFixed><<<num_sms * 4, 256, 0, st>>>(T * Hq, dqacc, static_cast<__nv_bfloat16*>(dq));
}

cudaError_t launch_bwd_finalize(const int32_t* cu, int n_docs, int64_t T, int Hq, int Hkv, int d, const void* dqacc,
                                void* dq, void* dk, void* dv, int num_sms, cudaStream_t st, uint64_t* dq_tag,
                                int rotate, int fixed) {
  if (fixed) launch_finalize_t<true>(cu, n_docs, T, Hq, Hkv, d, dqacc, dq, dk, dv, num_sms, st, dq_tag, rotate);
  else launch_finalize_t<false>(cu, n_docs, T, Hq, Hkv, d, dqacc, dq, dk, dv, num_sms, st, dq_tag, rotate);
  return cudaGetLastError();
}

}  // namespace flamia
