// Shared device helpers and layout constants of the MXFP8 attention kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace flamia {

constexpr int kTile = 128;       // query / key tile (rows of one MMA)
constexpr int kBlock = 32;       // token block, MX block, dS block edge
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Round-up shared exponent of a block whose maximum magnitude has fp32 bit
// pattern `amax_bits` (FLAMIA Section 3.2): the smallest E with
// amax <= 448 * 2^E, clamped to [-127, 127].  Writing amax = m 2^p with m in
// [1, 2): E = p - 8 + (m > 1.75).  448 = 1.75 * 2^8, and m > 1.75 exactly
// when the fp32 mantissa field exceeds 0x600000.  Subnormal fp32 maxima give
// p <= -127 and therefore clamp to -127, as does an all-zero block.
__device__ __forceinline__ int roundup_exponent_from_bits(uint32_t amax_bits) {
  const int expf = static_cast<int>(amax_bits >> 23);
  if (expf == 0) return -127;
  const int p = expf - 127;
  const int e = p - 8 + ((amax_bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^e as fp32 for e in [-126, 127] (exact).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Largest r in [0, n_docs) with cu[r] <= t (0 if none).  cu is non-decreasing.
__device__ __forceinline__ int find_doc(const int32_t* __restrict__ cu, int n_docs, int64_t t) {
  int lo = 0, hi = n_docs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(cu + mid)) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// ---------------------------------------------------------------- work plan
// The device-built schedule (FLAMIA Section 3.6.2): every document
// contributes nt = ceil(L/128) tiles per head, and a tile's cost c is the
// number of 128-blocks on the other side of the attention it visits,
// c in [1, nt].  Items are listed by decreasing cost.  Documents are sorted
// by decreasing nt, so the items of cost c are the first cnt_ge[c] documents
// of that order; bucket c starts at off[c] = sum_{c' > c} cnt_ge[c'].
struct PlanView {
  int32_t* hdr;          // [0] items per head, [1] max nt (C), [2] valid flag, [3] n_docs
  int32_t* sorted_docs;  // [n_docs]
  int32_t* cnt_ge;       // [C + 2]
  int32_t* off;          // [C + 2]
  int32_t* hist;         // [C + 2] scratch
  int32_t* fill;         // [C + 2] scratch
  int4* items;           // [items per head] records {doc, cost c, first token, length}
};

// Decode item u (0 <= u < items per head) into (doc, cost c).
__device__ __forceinline__ void plan_decode(const int32_t* __restrict__ off, const int32_t* __restrict__ sorted_docs,
                                            int C, int u, int& doc, int& c) {
  // smallest c in [1, C] with off[c] <= u (off is non-increasing in c)
  int lo = 1, hi = C;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(off + mid) <= u) hi = mid; else lo = mid + 1;
  }
  c = lo;
  doc = __ldg(sorted_docs + (u - __ldg(off + lo)));
}

// x * 2^e for e in [-254, 254], rounded once like ldexpf, without a branch:
// the power is applied as two factors 2^(e>>1) and 2^(e - (e>>1)), each a
// normal float.  For the factors used here (x = 1, or x = log2(e)/sqrt(d)
// within [2^-4, 1)) the first product is exact whenever the result is not
// zero, so only the second multiply rounds.  (pow2f(-127) reads as zero; it
// only occurs for e <= -253, where the result is zero anyway.)
__device__ __forceinline__ float scale_pow2(float x, int e) {
  const int e1 = e >> 1;
  return x * pow2f(e1) * pow2f(e - e1);
}

// Sylvester Hadamard transform of a 128-column row held by the 16 lanes of a
// half-warp (lane sub = lane % 16 holds columns 8 sub .. 8 sub + 7): radix-2
// butterflies (a, b) -> (a + b, a - b), lower element first, strides 1, 2, 4
// inside a lane and 8, 16, 32, 64 across lanes, in that order (FLAMIA
// Section 3.4, Appendix A.2).  Unnormalized: applying it twice multiplies by
// 128.  Every lane of the warp must call it.
__device__ __forceinline__ void fwht128_row(float (&x)[8], int sub) {
#pragma unroll
  for (int h = 1; h < 8; h *= 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 16; m *= 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = (sub & m) ? y - x[i] : x[i] + y;
    }
  }
}

// The same transform of a whole row held by one thread (n = 64 or 128).
template <int N>
__device__ __forceinline__ void fwht_inplace(float (&x)[N]) {
#pragma unroll
  for (int h = 1; h < N; h *= 2) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Snake walk over the longest-first item list: round k takes item
// k*G + b (k even) or k*G + G-1-b (k odd), alternating direction so long and
// short items spread over the grid.
struct SnakeIter {
  int k, b, G, total;
  __device__ __forceinline__ int next() {
    const long long g = (k & 1) ? (static_cast<long long>(k) * G + (G - 1 - b)) : (static_cast<long long>(k) * G + b);
    ++k;
    return g < total ? static_cast<int>(g) : -1;
  }
};

// Work items of one CTA in snake order over the device-built list, each
// item's record fetched one item ahead so the next decode finds it ready.
// `per` is the number of heads an item index covers (g = u * per + head).
struct ItemStream {
  SnakeIter it;
  const int4* items;
  int per;
  int g_next;
  int4 rec_next;
  __device__ __forceinline__ void start() {
    g_next = it.next();
    if (g_next >= 0) rec_next = __ldg(items + g_next / per);
  }
  // returns false at the end of the list
  __device__ __forceinline__ bool next(int& g, int4& rec) {
    g = g_next;
    rec = rec_next;
    if (g < 0) return false;
    g_next = it.next();
    if (g_next >= 0) rec_next = __ldg(items + g_next / per);
    return true;
  }
};

}  // namespace flamia
