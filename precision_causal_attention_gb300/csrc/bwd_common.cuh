// Work-item decoding and row stores shared by the backward kernels.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "flamia_common.cuh"
#include "launch.h"

namespace flamia {

struct BwdItem {
  int hk, doc, kt, nt, q0, n_it, group;
  int64_t s_doc;
  int L;
};

// item g = u * Hkv + hk with plan record rec = {doc, cost c, first token, length}
__device__ __forceinline__ BwdItem decode_bwd(const BwdArgs& a, int g, int4 rec) {
  BwdItem it;
  it.hk = g % a.Hkv;
  it.doc = rec.x;
  it.s_doc = rec.z;
  it.L = rec.w;
  it.nt = (it.L + kTile - 1) / kTile;
  const int c = rec.y;
  // causal: a key tile kt is seen by query tiles kt .. nt-1, cost nt - kt = c
  it.kt = a.causal ? it.nt - c : c - 1;
  it.q0 = a.causal ? it.kt : 0;
  it.group = a.Hq / a.Hkv;
  it.n_it = it.group * (it.nt - it.q0);
  return it;
}

// exact options helpers.  Round-up exponent of a positive finite fp32 value
// without the UE8M0 clamp (a zero or subnormal value gives a large negative
// number, below every block maximum), and 2^e as fp32 for any e: exact from
// 2^-149 to 2^127, 0 below, 2^127 above.
__device__ __forceinline__ int roundup_exponent_unclamped(uint32_t bits) {
  const int ef = static_cast<int>(bits >> 23);
  if (ef == 0) return -100000;
  return ef - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
}
__device__ __forceinline__ float pow2_any(int e) {
  if (e >= -126) return __int_as_float((min(e, 127) + 127) << 23);
  return e >= -149 ? __uint_as_float(1u << (e + 149)) : 0.f;
}

// iteration n of an item -> (query head, query tile)
__device__ __forceinline__ void bwd_iter(const BwdItem& w, int n, int& h, int& qt) {
  const int per_head = w.nt - w.q0;
  h = w.hk * w.group + n / per_head;
  qt = w.q0 + n % per_head;
}

// The same walk without division: query tiles q0 .. nt-1 of query head
// hk * group, then of the next head of the group.
struct BwdCursor {
  int h, qt;
  __device__ __forceinline__ void begin(const BwdItem& w) {
    h = w.hk * w.group;
    qt = w.q0;
  }
  __device__ __forceinline__ void advance(const BwdItem& w) {
    if (++qt == w.nt) {
      qt = w.q0;
      ++h;
    }
  }
};

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float* v, int n, float scale) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int k = 0; k < n / 8; ++k) {
    __nv_bfloat162 p0 = __floats2bfloat162_rn(v[8 * k + 0] * scale, v[8 * k + 1] * scale);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(v[8 * k + 2] * scale, v[8 * k + 3] * scale);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(v[8 * k + 4] * scale, v[8 * k + 5] * scale);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(v[8 * k + 6] * scale, v[8 * k + 7] * scale);
    d4[k] = make_uint4(*reinterpret_cast<uint32_t*>(&p0), *reinterpret_cast<uint32_t*>(&p1),
                       *reinterpret_cast<uint32_t*>(&p2), *reinterpret_cast<uint32_t*>(&p3));
  }
}

// 32 fp32 values given as bit patterns, times `scale`, stored as bf16.
__device__ __forceinline__ void store_row_bf16_bits(__nv_bfloat16* dst, const uint32_t (&r)[32], float scale) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(r[8 * k + 2 * j]) * scale,
                                               __uint_as_float(r[8 * k + 2 * j + 1]) * scale);
      w[j] = *reinterpret_cast<uint32_t*>(&p);
    }
    d4[k] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace flamia
