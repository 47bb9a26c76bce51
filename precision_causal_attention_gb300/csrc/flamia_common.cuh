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
  int32_t* hdr;          // [0] items per head, [1] max nt (C), [2] valid flag, [3] n_docs,
                         // [6] claim counter of the dynamic hand-out (zeroed with the plan)
  int32_t* sorted_docs;  // [n_docs]
  int32_t* cnt_ge;       // [C + 2]
  int32_t* off;          // [C + 2]
  int32_t* hist;         // [C + 2] scratch
  int32_t* fill;         // [C + 2] scratch
  int4* items;           // [items per head] records {doc, cost c, first token, length}
  // item order: 0 = by decreasing cost over all documents (bucket c holds one
  // item per document with nt >= c); 1 = document-major: documents by
  // decreasing nt, each document's tiles together in decreasing cost, so the
  // backward's dQ partials of one document arrive close together in time
  int order;
  int causal;            // order 1: how a record's cost field encodes the tile
  int32_t* doc_first;    // order 1: [n_docs] first item of each sorted document
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

// ---------------------------------------------------------------- work hand-out
// FLAMIA Section 3.6.2 hands the longest-first list out at run time.  The
// producer warp of every CTA claims the CTA's next item once it has issued
// the current item's last loads, and publishes it to the CTA's other warps
// through a ring of shared-memory slots: each slot has a full barrier (one
// arrival, the producer's) and an empty barrier (one arrival per consuming
// warp or thread).  Item -1 ends the stream.
//   dynamic (the default): a CTA's first item is its block index; every later
//     claim takes gridDim.x plus the old value of a global counter that the
//     plan job zeroed, so the longest items start first and each later one
//     goes to the first CTA that asks for work.
//   static: the snake walk above feeds the same ring.
// Which CTA computes an item changes no bit of its results: every item writes
// its own rows (the dQ reduce-adds are unordered either way).
constexpr int kItemSlots = 4;

struct ItemSlot {
  int4 rec;  // plan record {doc, cost c, first token, length}
  int g;     // item index (record u = g / per, head g % per); -1 = end
  int pad[3];
};

struct ItemRing {
  ItemSlot slot[kItemSlots];
  uint64_t full[kItemSlots];
  uint64_t empty[kItemSlots];
  // thread 0, before the CTA's first __syncthreads()
  __device__ __forceinline__ void init(uint32_t consumers) {
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], consumers);
    }
  }
};
static_assert(sizeof(ItemRing) == 192, "item ring layout");

// Producer side: every lane of the producer warp calls next() and publish()
// (lane 0 claims and writes; the results are warp-uniform).
struct ItemFeed {
  ItemRing* ring;
  const int4* items;
  int* counter;      // dynamic mode: the global claim counter
  int total, per;
  int dynamic;
  SnakeIter snake;
  int claimed, published;
  int* status;
  bool sleep = false;     // the slot waits sleep instead of polling
  // the next item index of this CTA (-1 at the end) and its record
  __device__ __forceinline__ int next(int4& rec) {
    int g = -1;
    if ((threadIdx.x & 31) == 0) {
      if (!dynamic) {
        g = snake.next();
      } else {
        const long long u = claimed == 0 ? static_cast<long long>(blockIdx.x)
                                         : static_cast<long long>(gridDim.x) + atomicAdd(counter, 1);
        g = u < total ? static_cast<int>(u) : -1;
      }
    }
    ++claimed;
    g = __shfl_sync(0xffffffffu, g, 0);
    rec = g >= 0 ? __ldg(items + g / per) : make_int4(0, 0, 0, 0);
    return g;
  }
  // hands item g to the consumers; false if a slot never came free (timeout)
  __device__ __forceinline__ bool publish(int g, int4 rec) {
    const int k = published++;
    const int s = k % kItemSlots;
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
      if (k >= kItemSlots) ok = mbar_wait(&ring->empty[s], ((k / kItemSlots) - 1) & 1, status, sleep);
      if (ok) {
        ring->slot[s].rec = rec;
        ring->slot[s].g = g;
        mbar_arrive(&ring->full[s]);
      }
    }
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  }
};

// Consumer side, for a whole warp (every lane calls next(); lane 0 waits and
// releases the slot) or a lone thread (whole_warp = false).  next() returns
// false at the end of the stream, or after a wait that timed out, which also
// raises the CTA's abort flag.
struct ItemReader {
  ItemRing* ring;
  volatile int* abort_flag;
  int* status;
  int taken;
  bool whole_warp;
  bool sleep = false;     // the slot waits sleep instead of polling
  __device__ __forceinline__ bool next(int& g, int4& rec) {
    if (*abort_flag) {
      g = -1;
      return false;
    }
    const int k = taken++;
    const int s = k % kItemSlots;
    const uint32_t par = (k / kItemSlots) & 1;
    bool ok;
    if (whole_warp) {
      int got = 0;
      if ((threadIdx.x & 31) == 0) got = mbar_wait(&ring->full[s], par, status, sleep) ? 1 : 0;
      __syncwarp();                                  // lane 0's acquire happens before the lanes' reads
      ok = __shfl_sync(0xffffffffu, got, 0) != 0;
    } else {
      ok = mbar_wait(&ring->full[s], par, status, sleep);
    }
    if (!ok) {
      *abort_flag = 1;
      g = -1;
      return false;
    }
    g = ring->slot[s].g;
    rec = ring->slot[s].rec;
    if (whole_warp) __syncwarp();
    if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive(&ring->empty[s]);
    return g >= 0;
  }
};

}  // namespace flamia
