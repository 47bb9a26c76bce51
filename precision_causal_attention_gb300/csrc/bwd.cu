// MXFP8 causal packed attention backward for sm_103a.
//
// Method: FLAMIA (arXiv 2611.03344) Sections 2, 3.1, 3.3, 3.5.3 and
// Appendix B.1.  One CTA owns one 128-key tile of one document for one
// key/value head and loops over the query tiles that see it, for every
// query head of the grouped-query group:
//   S  = Qhat Khat^T          unscaled E4M3 MMA, same operands, shape, K order
//                             and scale folding as the forward, so the score
//                             tile is bitwise the forward's
//   P  = 2^(S2 - LSE2)        S2 = acc * 2^{E_Q+E_K} log2(e)/sqrt(d), fp32, MUFU
//   dP = dOhat Vhat^T         unscaled MMA, token-block factors folded in
//   dS = P o (dP - D)         fp32; quantized per 32x32 (query, key) block with
//                             the round-up exponent: one payload serves both
//                             dQ (contraction over keys) and dK (over queries)
//   dV += P'^T dOhat          P' = E4M3(2^8 P), scale 2^-8; block-scaled MMA
//   dK += dShat^T Qhat        block-scaled MMA (MN-major operands from the
//                             same shared-memory tiles)
//   dQ  = dShat Khat          block-scaled MMA, staged in shared memory and
//                             added into the fp32 dQ accumulator with TMA bulk
//                             reduce-adds (1/sqrt(d) applied at finalisation)
// dK and dV accumulate in tensor memory across the loop and are written once.
//
// This kernel serves d = 128, and d = 64 with the exact options
// (bwd_kernel<64, true>; Section 3.2 and Appendix A.3); the default d = 64
// path has its own kernel with eight compute warps and a deeper MMA schedule
// (bwd_d64.cu).  With the exact options, Q, K, V and dO carry per-token
// exponents:
//   * S and dP are block-scaled MMAs with K's and V's per-key scales;
//   * P' carries the row's dO exponent against the largest of its 32-query
//     block, whose exponent becomes the dV operand's scale;
//   * dK reads a 32 x 32-block payload of dS times the row's Q exponent;
//   * dQ reads a second payload: dS times K's per-key exponent, with one
//     exponent per (query row, 32-key group);
//   * dQ, dK and dV read K, Q and dO codes with scale 1.
//
// Warp roles (320 threads, one CTA per SM, 512 TMEM columns):
//   compute    warps 0-7: warp w reads TMEM lanes 32 (w % 4) .. + 31, the
//              query rows of S/dP/dQ and the key rows of dV/dK; warpgroup
//              c = w / 4 takes key columns [64c, 64c + 64) of S and dP and
//              columns [64c, 64c + 64) of dQ when draining it, and the first
//              warpgroup writes the item's dV and dK rows and the exact
//              options' per-item fold tables.
//   next warp  TMA producer: K/V once per item, Q/dO through a 2-stage ring,
//              plus the block-scale words the producer can derive from the
//              token scale tables
//   last warp  MMA issuer (lane 0) and TMEM owner
// TMEM, d = 64:  S [0,128) dP [128,256) dV [256,320) dK [320,384) dQ [384,448)
//                scale factors [448,472)
//       d = 128: dV [0,128) dK [128,256) S [256,384) dP [384,512); dQ reuses
//                the S columns and the scale factors sit in the dP columns,
//                both free once the compute warps have read S and dP.
#include <cuda_bf16.h>
#include <cstdint>

#include "bwd_common.cuh"

namespace flamia {

template <int D, bool kExact = false, bool kF4 = false>
struct BwdLayout {
  static constexpr int kStages = 2;
  static constexpr int kTileBytes = kTile * D;
  static constexpr uint32_t kSwz = (D == 64) ? kSwizzle64B : kSwizzle128B;
  // shared memory
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;                  // kStages tiles
  static constexpr int kDO = kQ + kStages * kTileBytes;       // kStages tiles
  static constexpr int kPp = kDO + kStages * kTileBytes;      // P' codes [128 q][128 k], 128B swizzle
  static constexpr int kDS = kPp + kTile * kTile;             // dS codes [128 q][128 k]
  static constexpr int kSfaDV = kDS + kTile * kTile;          // 512 B each
  static constexpr int kSfaDK = kSfaDV + 512;
  static constexpr int kSfaDQ = kSfaDK + 512;
  static constexpr int kSfbDQ = kSfaDQ + 512;
  static constexpr int kSfbDV = kSfbDQ + 512;                 // per stage
  static constexpr int kSfbDK = kSfbDV + kStages * 512;       // per stage
  // dQ staging for the bulk reduce-add: per buffer d/32 boxes of 128 rows x 32 fp32 (128B swizzle)
  static constexpr int kDqBufs = (D == 64) ? 2 : 1;
  static constexpr int kDqBufBytes = D * kTile * 4;
  // deterministic option: the same area as kDetSlots slots of 128 rows x
  // kDetRowBytes (32 fixed-point columns per row, padded so consecutive rows
  // start in different banks)
  static constexpr int kDetRowBytes = 256;   // unpadded with two slots, to fit the budget
  static constexpr int kDetSlotBytes = kTile * kDetRowBytes;
  // compute warps: eight, two warpgroups, warpgroup c taking key columns
  // [64c, 64c + 64) of S and dP and the same half of dQ's columns
  static constexpr bool kSplit = true;
  // the exact options issue an iteration's dQ MMA before its dV and dK MMAs,
  // so the dQ drain overlaps them (measured: 3.66 -> 3.40 ms on a 16384-token
  // document; the default path is 1.6 % slower that way and keeps dQ last)
  static constexpr bool kDqFirst = kExact;
  static constexpr int kComputeWarps = kSplit ? 8 : 4;
  static constexpr int kThreads = 32 * (kComputeWarps + 2);
  static constexpr int kWProd = kComputeWarps, kWMma = kComputeWarps + 1;
  // the deterministic option stages one padded row per compute thread
  static constexpr int kDetSlots = kSplit ? 2 : 1;
  static constexpr int kDqRegion = kDetSlots * kDetSlotBytes > kDqBufs * kDqBufBytes ? kDetSlots * kDetSlotBytes
                                                                                      : kDqBufs * kDqBufBytes;
  static constexpr int kDQs = (kSfbDK + kStages * 512 + 1023) / 1024 * 1024;
  // exact options: the dQ payload of dS (per-row exponents, K fold), the
  // scale words of the S and dP MMAs (Q and dO: constant 1; K and V: per key)
  // and the K fold table (fp32 2^(E_K(j) - G_g) per key, G_g per group)
  static constexpr int kDS2 = (kDQs + kDqRegion + 1023) / 1024 * 1024;
  static constexpr int kSa1 = kDS2 + kTile * kTile;
  static constexpr int kSfbS = kSa1 + 512;
  static constexpr int kSfbP = kSfbS + 512;
  static constexpr int kFk = kSfbP + 512;
  static constexpr int kGk = kFk + 512;
  // d = 128: the V fold table (fp32 2^(E_V(j) - Gv_g) per key, Gv_g per
  // group), for the per-column factors of dP
  static constexpr int kFv = kGk + 512;
  static constexpr int kGv = kFv + 512;
  // NVFP4 option: the 4-bit Q tile of each stage and K tile of the item for
  // the recomputed S, and the scale words of the 4-bit S MMA (Q per stage,
  // K per item; one 512-byte block per 64-element chunk)
  static constexpr int kC4 = D / 64;
  static constexpr int kQ4 = (kDQs + kDqRegion + 1023) / 1024 * 1024;
  static constexpr int kK4 = kQ4 + kStages * (kTileBytes / 2);
  static constexpr int kSq4 = kK4 + kTileBytes / 2;
  static constexpr int kSk4 = kSq4 + kStages * kC4 * 512;
  static constexpr int kBar = kExact ? kGv + 512 : (kF4 ? kSk4 + kC4 * 512 : kDQs + kDqRegion);
  enum {
    bKVFull = 0,
    bKVEmpty,
    bQDFull,
    bQDEmpty = bQDFull + kStages,
    bSdpFull = bQDEmpty + kStages,
    bSdpEmpty,
    bDsFull,
    bDsEmpty,
    bDqFull,
    bDqEmpty,
    bAccEmpty,
    bFinal,
    bFkReady,                  // exact options: the K fold table of an item is written
    bStageFree,                // the dQ staging buffer's previous reduce-add has read it (one arrival)
    bStaged,                   // every compute thread has staged its dQ rows
    bSDone,                    // NVFP4 option at d = 128: S complete before dP overwrites its scale columns
    kNumBars
  };
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 8;
  static constexpr int kRing = (kAbort + 16 + 15) / 16 * 16;   // work hand-out ring (ItemRing)
  static constexpr int kBytes = kRing + static_cast<int>(sizeof(ItemRing));
  static constexpr int kSmemAlloc = kBytes + 1024;
  // tensor memory columns
  static constexpr uint32_t kTS = (D == 64) ? 0 : 256;
  static constexpr uint32_t kTdP = (D == 64) ? 128 : 384;
  static constexpr uint32_t kTdV = (D == 64) ? 256 : 0;
  static constexpr uint32_t kTdK = (D == 64) ? 320 : 128;
  static constexpr uint32_t kTdQ = (D == 64) ? 384 : 256;
  static constexpr uint32_t kTSf = (D == 64) ? 448 : 384;
  static constexpr uint32_t kTSfaDV = kTSf + 0;
  static constexpr uint32_t kTSfbDV = kTSf + 4;
  static constexpr uint32_t kTSfaDK = kTSf + 8;
  static constexpr uint32_t kTSfbDK = kTSf + 12;
  static constexpr uint32_t kTSfaDQ = kTSf + 16;
  static constexpr uint32_t kTSfbDQ = kTSf + 20;
  // exact options at d = 64, where TMEM has room: S/dP scale factors.  At
  // d = 128 the S and dP columns take the whole rest of TMEM, so S and dP
  // stay unscaled MMAs and K's and V's per-key exponents are applied as fp32
  // column factors by the compute warps (kFoldCols).
  static constexpr uint32_t kTSa1 = kTSf + 24;
  static constexpr uint32_t kTSbS = kTSf + 28;
  static constexpr uint32_t kTSbP = kTSf + 32;
  static constexpr bool kFoldCols = kExact && D == 128;
  static_assert(!kExact || D == 128 || kTSbP + 4 <= 512, "tensor memory budget");
  // NVFP4 option: the 4-bit S MMA's scale factors (Q per stage, K per item).
  // At d = 128 they sit in the dP columns, so S completes before dP is issued.
  static constexpr uint32_t kTSq4 = (D == 64) ? kTSf + 24 : 448;
  static constexpr uint32_t kTSk4 = kTSq4 + kStages * 4 * kC4;
  static_assert(!kF4 || kTSk4 + 4 * kC4 <= 512, "tensor memory budget");
  static_assert(!(kF4 && kExact), "the NVFP4 path and the exact options are separate");
  static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
  static constexpr float kSmScale = (D == 64) ? 0.18033688011112042f : 0.12751743082459868f;
  static constexpr float kInvSqrtD = (D == 64) ? 0.125f : 0.08838834764831845f;
};

template <int D, bool kExact, bool kDump = false, bool kF4 = false>
__global__ void __launch_bounds__(BwdLayout<D, kExact, kF4>::kThreads, 1) bwd_kernel(const __grid_constant__ BwdArgs a) {
  using Lay = BwdLayout<D, kExact, kF4>;
  // the producer sleeps in its waits (it runs well ahead of the MMAs); the
  // other roles poll (sleeping changed the backward's time by under 1 %)
  constexpr unsigned kSleepMask = kRoleProducer;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Lay::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars[Lay::bKVFull], 1);
    mbar_init(&bars[Lay::bKVEmpty], 1);
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&bars[Lay::bQDFull + s], 1);
      mbar_init(&bars[Lay::bQDEmpty + s], 1);
    }
    constexpr uint32_t kCT = 32 * Lay::kComputeWarps;     // compute threads
    mbar_init(&bars[Lay::bSdpFull], 1);
    mbar_init(&bars[Lay::bSdpEmpty], kCT);
    mbar_init(&bars[Lay::bDsFull], kCT);
    mbar_init(&bars[Lay::bDsEmpty], 1);
    mbar_init(&bars[Lay::bDqFull], 1);
    mbar_init(&bars[Lay::bDqEmpty], kCT);
    mbar_init(&bars[Lay::bAccEmpty], 128);                // the first warpgroup writes dV, dK
    mbar_init(&bars[Lay::bFinal], 1);
    mbar_init(&bars[Lay::bFkReady], kCT);
    mbar_init(&bars[Lay::bStageFree], 1);
    mbar_init(&bars[Lay::bStaged], kCT);
    mbar_init(&bars[Lay::bSDone], 1);
    // consumers of the item ring: the compute warps and the MMA issuer
    reinterpret_cast<ItemRing*>(smem + Lay::kRing)->init(Lay::kComputeWarps + 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == Lay::kWMma) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (warp == Lay::kWProd && lane == 0) {
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
    tma_prefetch_desc(&a.tm_do);
    tma_prefetch_desc(&a.tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  const int valid_plan = __ldg(a.plan_hdr + 2);
  const int total = valid_plan ? __ldg(a.plan_hdr + 0) * a.Hkv : 0;
  ItemRing* ring = reinterpret_cast<ItemRing*>(smem + Lay::kRing);
  // every role reads its items from the ring the producer fills
  ItemReader work{ring, abort_flag, a.status, 0, true};
  const int64_t T = a.T;

  if (warp < Lay::kComputeWarps) {
    // ------------------------------------------------------------ compute
    work.sleep = role_sleeps(kSleepMask, kRoleCompute);
    const int quad = warp & 3;                       // TMEM lanes 32 quad .. + 31
    const int half = Lay::kSplit ? (warp >> 2) : 0;  // key columns [64 half, + 64) when split
    constexpr int kNG = Lay::kSplit ? 2 : 4;         // 32-key groups per thread
    const int row = 32 * quad + lane;                // TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
    uint8_t* sPp = smem + Lay::kPp;
    uint8_t* sDS = smem + Lay::kDS;
    const uint32_t rbase = (row >> 3) * 1024 + (row & 7) * 128;
    int it = 0, items_c = 0;
    bool ok = true;
    for (;;) {
      int g;
      int4 rec;
      if (!work.next(g, rec) || *abort_flag) break;
      const BwdItem w = decode_bwd(a, g, rec);
      if constexpr (kExact) {
        // K fold table of this key tile: thread row owns key row (group =
        // quad).  The previous item's readers are past their last dS: this
        // thread waited for that item's last dq_full, and the dQ MMA follows
        // every compute thread's ds_full arrival.
        const int kj = w.kt * kTile + row;
        const int kb = kj < w.L ? static_cast<int>(__ldg(a.k_scales + static_cast<int64_t>(w.hk) * T + w.s_doc + kj)) : -1;
        const int gmax = max(__reduce_max_sync(0xffffffffu, kb), 0);
        // (the first warpgroup writes the tables, both read them)
        if (half == 0) reinterpret_cast<float*>(smem + Lay::kFk)[row] = kb >= 0 ? pow2_any(kb - gmax) : 0.f;
        if (half == 0 && lane == 0) reinterpret_cast<int*>(smem + Lay::kGk)[quad] = gmax;
        if constexpr (Lay::kFoldCols) {
          // the same table for V (dP's per-column factors)
          const int vb = kj < w.L ? static_cast<int>(__ldg(a.v_scales + static_cast<int64_t>(w.hk) * T + w.s_doc + kj)) : -1;
          const int gvmax = max(__reduce_max_sync(0xffffffffu, vb), 0);
          if (half == 0) reinterpret_cast<float*>(smem + Lay::kFv)[row] = vb >= 0 ? pow2_any(vb - gvmax) : 0.f;
          if (half == 0 && lane == 0) reinterpret_cast<int*>(smem + Lay::kGv)[quad] = gvmax;
        }
        mbar_arrive(&bars[Lay::bFkReady]);
        if (!mbar_wait(&bars[Lay::bFkReady], items_c & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
      }
      ++items_c;
      int ek[4], ev[4];
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int rel = w.kt * kTile + gg * kBlock;
        const bool in = rel < w.L;
        const int64_t tk = static_cast<int64_t>(w.hk) * T + w.s_doc + rel;
        ek[gg] = in ? static_cast<int>(__ldg(a.k_scales + tk)) - 127 : 0;
        ev[gg] = in ? static_cast<int>(__ldg(a.v_scales + tk)) - 127 : 0;
      }
      // per-row scalars of iteration n (scales, LSE, D), loaded one iteration ahead
      // Raw values are loaded unconditionally (index clamped into the
      // document) and only converted when used, so the loads issued one
      // iteration ahead do not stall the warp at the point of issue.
      struct RowVals { uint32_t eqb, edob; float lse, Di; };
      auto load_row = [&](int n) {
        RowVals v;
        int h, qt;
        bwd_iter(w, n, h, qt);
        const int qi = min(qt * kTile + row, w.L - 1);
        const int64_t ht = static_cast<int64_t>(h) * T + w.s_doc + qi;
        v.eqb = __ldg(a.q_scales + ht);
        v.edob = __ldg(a.do_scales + ht);
        v.lse = __ldg(a.lse + ht);
        v.Di = __ldg(a.D + ht);
        return v;
      };
      RowVals rv_next = load_row(0);
      for (int n = 0; n < w.n_it; ++n, ++it) {
        int h, qt;
        bwd_iter(w, n, h, qt);
        const int qi = qt * kTile + row;
        const bool valid = qi < w.L;
        const int64_t t = w.s_doc + qi;
        const RowVals rv = rv_next;
        if (n + 1 < w.n_it) rv_next = load_row(n + 1);
        // A row past the document end is zeroed through its exponent offset
        // (arg_add = -inf gives P = 0, P' = 0 and dS = 0 in every column), so
        // it needs no column mask.
        int nvis;
        if (!valid) nvis = kTile;
        else if (a.causal) nvis = (qt == w.kt) ? row + 1 : kTile;
        else nvis = min(kTile, w.L - w.kt * kTile);
        const bool full = __all_sync(0xffffffffu, nvis == kTile);
        // 2^8 P = 2^(S2 - LSE2 + 8): the dV operand directly; dS is carried as
        // 2^8 dS, the factor leaving the block exponent exactly
        const float arg_add = valid ? 8.f - rv.lse * kLog2e : -INFINITY;
        const int r_eq = valid ? static_cast<int>(rv.eqb) - 127 : 0;
        const int r_edo = valid ? static_cast<int>(rv.edob) - 127 : 0;
        const float negD = valid ? -rv.Di : 0.f;

        if (!mbar_wait(&bars[Lay::bSdpFull], it & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
        // the previous iteration's dV/dK MMAs must be done with the P'/dS tiles
        if (it > 0 && !mbar_wait(&bars[Lay::bDsEmpty], (it - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
        tc_fence_after();
        int Eds[4], Edq[4];
        // exact options: dV's operand E4M3(2^8 P 2^(E_dO(i) - H_b)) carries the
        // row's dO exponent relative to sigma_b = max(H_b - 8, -127), H_b the
        // largest dO exponent among the document rows of this warp's 32-query
        // block; sigma_b is the block's scale along the dV contraction
        float fo = 1.f;
        if constexpr (kExact) {
          const int hb = __reduce_max_sync(0xffffffffu, valid ? r_edo : -100000);
          const int sig = max(hb - 8, -127);
          if (valid) fo = pow2_any(r_edo - sig - 8);
          uint8_t* dv_bytes = smem + Lay::kSfaDV;
          if (half == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) dv_bytes[(lane * 4 + i) * 4 + quad] = static_cast<uint8_t>(sig + 127);
          }
        }
#pragma unroll
        for (int j = 0; j < kNG; ++j) {
          const int gg = kNG * half + j;                 // the 32-key group
          uint32_t sa[32], pa[32];
          // the group's S and dP columns, one wait for both loads
          tmem_ld32x2_sync(tbase + lane_base + Lay::kTS + 32 * gg, sa, tbase + lane_base + Lay::kTdP + 32 * gg, pa);
          // exact options: K's and V's per-key scales are applied in the MMAs
          // (d = 64), or as column factors 2^(E(j) - G_g) with the group's
          // largest exponent G_g in the row factor (d = 128).  acc 2^(E(j) -
          // G_g) is exact, so S2 and dP round once, to the same values as
          // with the scales inside the MMA.
          int gk_e = kExact ? 0 : ek[gg], gv_e = kExact ? 0 : ev[gg];
          if constexpr (Lay::kFoldCols) {
            gk_e = reinterpret_cast<const int*>(smem + Lay::kGk)[gg] - 127;
            gv_e = reinterpret_cast<const int*>(smem + Lay::kGv)[gg] - 127;
            const float4* fk4 = reinterpret_cast<const float4*>(smem + Lay::kFk) + 8 * gg;
            const float4* fv4 = reinterpret_cast<const float4*>(smem + Lay::kFv) + 8 * gg;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 fk = fk4[u], fv = fv4[u];
              sa[4 * u] = __float_as_uint(__uint_as_float(sa[4 * u]) * fk.x);
              sa[4 * u + 1] = __float_as_uint(__uint_as_float(sa[4 * u + 1]) * fk.y);
              sa[4 * u + 2] = __float_as_uint(__uint_as_float(sa[4 * u + 2]) * fk.z);
              sa[4 * u + 3] = __float_as_uint(__uint_as_float(sa[4 * u + 3]) * fk.w);
              pa[4 * u] = __float_as_uint(__uint_as_float(pa[4 * u]) * fv.x);
              pa[4 * u + 1] = __float_as_uint(__uint_as_float(pa[4 * u + 1]) * fv.y);
              pa[4 * u + 2] = __float_as_uint(__uint_as_float(pa[4 * u + 2]) * fv.z);
              pa[4 * u + 3] = __float_as_uint(__uint_as_float(pa[4 * u + 3]) * fv.w);
            }
          }
          // (the NVFP4 path's Q and K scales are inside the S MMA)
          const float cg = kF4 ? Lay::kSmScale
                               : scale_pow2(a.hadamard ? Lay::kSmScale * (1.f / D) : Lay::kSmScale, r_eq + gk_e);
          const float cdp = scale_pow2(1.f, r_edo + gv_e);
          if constexpr (kDump) {
            // diagnostic copy of the recomputed raw S tile and the group factors
            if (w.doc == a.dump.doc && w.kt == a.dump.kt && h == a.dump.h && qt == a.dump.qt) {
#pragma unroll
              for (int c = 0; c < 32; ++c) a.dump.s[row * kTile + 32 * gg + c] = __uint_as_float(sa[c]);
              a.dump.f[row * 4 + gg] = cg;
            }
          }
          float ds[32];
          uint32_t pw[8];
          float amax = 0.f;
          if (full) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float a0, a1, t0, t1;
              ffma2(a0, a1, __uint_as_float(sa[c]), __uint_as_float(sa[c + 1]), cg, cg, arg_add, arg_add);
              const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
              ffma2(t0, t1, __uint_as_float(pa[c]), __uint_as_float(pa[c + 1]), cdp, cdp, negD, negD);
              fmul2(ds[c], ds[c + 1], p0, p1, t0, t1);
              amax = max3f(amax, fabsf(ds[c]), fabsf(ds[c + 1]));
              const uint32_t pc = kExact ? cvt_e4m3x2(p0 * fo, p1 * fo) : cvt_e4m3x2(p0, p1);
              if ((c & 2) == 0) pw[c >> 2] = pc; else pw[c >> 2] |= pc << 16;
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const int col = 32 * gg + c;
              const float p0 = (col < nvis) ? ex2_approx(fmaf(__uint_as_float(sa[c]), cg, arg_add)) : 0.f;
              const float p1 = (col + 1 < nvis) ? ex2_approx(fmaf(__uint_as_float(sa[c + 1]), cg, arg_add)) : 0.f;
              ds[c] = (col < nvis) ? p0 * fmaf(__uint_as_float(pa[c]), cdp, negD) : 0.f;
              ds[c + 1] = (col + 1 < nvis) ? p1 * fmaf(__uint_as_float(pa[c + 1]), cdp, negD) : 0.f;
              amax = max3f(amax, fabsf(ds[c]), fabsf(ds[c + 1]));
              const uint32_t pc = kExact ? cvt_e4m3x2(p0 * fo, p1 * fo) : cvt_e4m3x2(p0, p1);
              if ((c & 2) == 0) pw[c >> 2] = pc; else pw[c >> 2] |= pc << 16;
            }
          }
          // 32x32 block of dS: this warp's 32 query rows x these 32 keys.  The
          // exponent of 2^8 dS is 8 more than that of dS (clamped at -127).
          float inv;
          if constexpr (kExact) {
            // dK payload: y = dS 2^E_Q(i) = ds 2^(E_Q(i) - 8) in 32x32 blocks
            const int et = amax > 0.f ? roundup_exponent_unclamped(__float_as_uint(amax)) + r_eq - 8 : -100000;
            const int E = min(max(__reduce_max_sync(0xffffffffu, et), -127), 127);
            Eds[gg] = E;
            inv = pow2_any(r_eq - 8 - E);
          } else {
            const int E8 = roundup_exponent_from_bits(warp_max_u32(__float_as_uint(amax)));
            const int E = E8 - 8 < -127 ? -127 : E8 - 8;
            Eds[gg] = E;
            const int sh = E + 8 > 126 ? 126 : E + 8;
            inv = pow2f(-sh);
          }
          uint32_t dw[8];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            float s0, s1, s2, s3;
            fmul2(s0, s1, ds[c], ds[c + 1], inv, inv);
            fmul2(s2, s3, ds[c + 2], ds[c + 3], inv, inv);
            dw[c >> 2] = cvt_e4m3x4(s0, s1, s2, s3);
          }
          if constexpr (kExact) {
            // dQ payload (K fold, per-query-row exponent): x = dS 2^E_K(j),
            // computed as x' = ds 2^(E_K(j) - G_g), so x = x' 2^(G_g - 135)
            // with G_g the group's largest K scale byte
            const float4* fk4 = reinterpret_cast<const float4*>(smem + Lay::kFk) + 8 * gg;
            float xs[32];
            float ax = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 f = fk4[u];
              fmul2(xs[4 * u], xs[4 * u + 1], ds[4 * u], ds[4 * u + 1], f.x, f.y);
              fmul2(xs[4 * u + 2], xs[4 * u + 3], ds[4 * u + 2], ds[4 * u + 3], f.z, f.w);
              ax = max3f(ax, fabsf(xs[4 * u]), fabsf(xs[4 * u + 1]));
              ax = max3f(ax, fabsf(xs[4 * u + 2]), fabsf(xs[4 * u + 3]));
            }
            const int gk = reinterpret_cast<const int*>(smem + Lay::kGk)[gg];
            const int eq_ = ax > 0.f ? roundup_exponent_unclamped(__float_as_uint(ax)) + gk - 135 : -127;
            const int Eq = min(max(eq_, -127), 127);
            Edq[gg] = Eq;
            const float invq = pow2_any(gk - 135 - Eq);
            uint32_t qw[8];
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              float s0, s1, s2, s3;
              fmul2(s0, s1, xs[c], xs[c + 1], invq, invq);
              fmul2(s2, s3, xs[c + 2], xs[c + 3], invq, invq);
              qw[c >> 2] = cvt_e4m3x4(s0, s1, s2, s3);
            }
            uint8_t* sDS2 = smem + Lay::kDS2;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int k = 2 * gg + hf;
              const uint32_t off = rbase + ((k ^ (row & 7)) << 4);
              *reinterpret_cast<uint4*>(sDS2 + off) = make_uint4(qw[4 * hf], qw[4 * hf + 1], qw[4 * hf + 2], qw[4 * hf + 3]);
            }
          } else {
            Edq[gg] = Eds[gg];
          }
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int k = 2 * gg + hf;
            const uint32_t off = rbase + ((k ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(sPp + off) = make_uint4(pw[4 * hf], pw[4 * hf + 1], pw[4 * hf + 2], pw[4 * hf + 3]);
            *reinterpret_cast<uint4*>(sDS + off) = make_uint4(dw[4 * hf], dw[4 * hf + 1], dw[4 * hf + 2], dw[4 * hf + 3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&bars[Lay::bSdpEmpty]);
        // block-scale words of dS.  dQ = dS K contracts over keys: query row
        // 32w + r reads byte g = E(w, g).  dK = dS^T Q contracts over queries:
        // key row 32i + r reads byte w = E(w, i).
        {
          uint32_t word = 0;
#pragma unroll
          for (int j = 0; j < kNG; ++j) word |= static_cast<uint32_t>(Edq[kNG * half + j] + 127) << (8 * j);
          if constexpr (Lay::kSplit)      // bytes 2 half, 2 half + 1 of the row's word
            reinterpret_cast<uint16_t*>(smem + Lay::kSfaDQ)[(lane * 4 + quad) * 2 + half] = static_cast<uint16_t>(word);
          else
            reinterpret_cast<uint32_t*>(smem + Lay::kSfaDQ)[lane * 4 + quad] = word;
          uint8_t* dk_bytes = smem + Lay::kSfaDK;
#pragma unroll
          for (int j = 0; j < kNG; ++j) {
            const int i = kNG * half + j;
            dk_bytes[(lane * 4 + i) * 4 + quad] = static_cast<uint8_t>(Eds[i] + 127);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[Lay::bDsFull]);

        // dQ partial of this (key tile, query tile): staged in shared memory
        // and added to the fp32 accumulator with a TMA bulk reduce-add.  Rows
        // of the tile outside the document carry exact zeros (their dS row is
        // zero), and adding a zero leaves the accumulator bits unchanged.
        if (!mbar_wait(&bars[Lay::bDqFull], it & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
        tc_fence_after();
        if (a.det_dq) {
          // Deterministic option: each partial becomes a 64-bit fixed-point
          // integer and every thread adds its own query row with integer bulk
          // reduce-adds (32 columns per pass, one padded staging row per
          // thread), so the sum does not depend on the order in which key
          // tiles arrive.  Rows outside the document are skipped; each
          // thread's staging row is its own.
          unsigned long long* grow = reinterpret_cast<unsigned long long*>(a.dqacc) + (t * a.Hq + h) * D;
          // this warpgroup's 32-column blocks of the row
          constexpr int kCB = (D / 32) / (Lay::kSplit ? 2 : 1);
#pragma unroll 1
          for (int cc = kCB * half; cc < kCB * half + kCB; ++cc) {
            uint32_t r[32];
            tmem_ld32_sync(tbase + lane_base + Lay::kTdQ + 32 * cc, r);
            uint8_t* slot = smem + Lay::kDQs + half * Lay::kDetSlotBytes + row * Lay::kDetRowBytes;
            bulk_wait_group_read<0>();                     // this thread's previous reduce has read its row
#pragma unroll
            for (int k = 0; k < 16; ++k)
              *reinterpret_cast<ulonglong2*>(slot + 16 * k) =
                  make_ulonglong2(dq_fixed(__uint_as_float(r[2 * k])), dq_fixed(__uint_as_float(r[2 * k + 1])));
            fence_proxy_async_smem();
            if (valid) bulk_reduce_add_u64(grow + 32 * cc, slot, 256);
            bulk_commit_group();
          }
          tc_fence_before();
          mbar_arrive(&bars[Lay::bDqEmpty]);
        } else {
          // The staging buffer is shared: thread 0 frees it (its previous
          // reduce-add has read it) and issues the next one once every compute
          // thread has staged its rows; both handshakes are bounded mbarrier
          // waits, one phase per iteration.
          uint8_t* stage = smem + Lay::kDQs + (it % Lay::kDqBufs) * Lay::kDqBufBytes;
          if (threadIdx.x == 0) {
            bulk_wait_group_read<Lay::kDqBufs - 1>();
            mbar_arrive(&bars[Lay::bStageFree]);
          }
          if (!mbar_wait(&bars[Lay::bStageFree], it & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
          // this warpgroup's 32-column boxes, two per TMEM wait
          constexpr int kCB = (D / 32) / (Lay::kSplit ? 2 : 1);
#pragma unroll
          for (int cc = kCB * half; cc < kCB * half + kCB; cc += 2) {
            uint32_t r0[32], r1[32];
            tmem_ld32x2_sync(tbase + lane_base + Lay::kTdQ + 32 * cc, r0, tbase + lane_base + Lay::kTdQ + 32 * cc + 32, r1);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t (&r)[32] = u ? r1 : r0;
              uint8_t* box = stage + (cc + u) * (kTile * 128) + row * 128;
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4*>(box + ((k ^ (row & 7)) << 4)) =
                    make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
            }
          }
          tc_fence_before();
          mbar_arrive(&bars[Lay::bDqEmpty]);
          fence_proxy_async_smem();
          mbar_arrive(&bars[Lay::bStaged]);
          if (threadIdx.x == 0) {
            if (!mbar_wait(&bars[Lay::bStaged], it & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
            const int32_t y = static_cast<int32_t>(w.s_doc + qt * kTile);
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) tma_reduce_add_2d(&a.tm_dq, h * D + 32 * cc, y, stage + cc * (kTile * 128));
            bulk_commit_group();
          }
        }
      }
      if (!ok) break;
      // item epilogue: dV, dK rows (TMEM lane = key row), written by the first
      // warpgroup (the Hadamard option's inverse rotation needs whole rows),
      // once the item's last dV and dK MMAs have completed: dq_full of its
      // last iteration implies it when dQ is issued last, ds_empty otherwise
      if (half != 0) continue;
      if constexpr (Lay::kDqFirst) {
        if (!mbar_wait(&bars[Lay::bDsEmpty], (it - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      float acc[D];
      const int kj = w.kt * kTile + row;
      const bool kvalid = kj < w.L;
      __nv_bfloat16* dv_row = a.dv + ((w.s_doc + kj) * a.Hkv + w.hk) * D;
      __nv_bfloat16* dk_row = a.dk + ((w.s_doc + kj) * a.Hkv + w.hk) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32_sync(tbase + lane_base + Lay::kTdV + 32 * cc, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[32 * cc + k] = __uint_as_float(r[k]);
      }
      if (kvalid) store_row_bf16(dv_row, acc, D, 1.f);
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        tmem_ld32_sync(tbase + lane_base + Lay::kTdK + 32 * cc, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[32 * cc + k] = __uint_as_float(r[k]);
      }
      tc_fence_before();
      mbar_arrive(&bars[Lay::bAccEmpty]);
      // Hadamard option: dK of the rotated K, mapped back by H_d / d
      if (a.hadamard) fwht_inplace<D>(acc);
      if (kvalid) store_row_bf16(dk_row, acc, D, a.hadamard ? Lay::kInvSqrtD * (1.f / D) : Lay::kInvSqrtD);
    }
    if (!ok) *abort_flag = 1;
    // every reduce-add has landed before the CTA exits (the deterministic
    // option's are issued by every thread)
    if (a.det_dq || threadIdx.x == 0) bulk_wait_group<0>();
  } else if (warp == Lay::kWProd) {
    // ------------------------------------------------------------ TMA producer
    int it = 0, items = 0, kv_issued = 0;
    ItemFeed feed{ring, a.plan_items, a.item_counter, total, a.Hkv, a.schedule == 0,
                  SnakeIter{0, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total}, 0, 0, a.status, role_sleeps(kSleepMask, kRoleProducer)};
    int4 rec;
    int g = feed.next(rec);
    bool ok = feed.publish(g, rec);
    while (ok && g >= 0 && !*abort_flag) {
      const BwdItem w = decode_bwd(a, g, rec);
      if (items > 0 && !mbar_wait(&bars[Lay::bKVEmpty], (items - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleProducer))) { ok = false; break; }
      if constexpr (kExact) {
        // K's codes enter dQ with scale 1 (their exponents are folded into
        // dS); S and dP take K's and V's per-key scales: row r, word i = the
        // scale byte of key 32 i + r
        reinterpret_cast<uint4*>(smem + Lay::kSfbDQ)[lane] = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
        uint32_t kw[4], vw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rel = w.kt * kTile + 32 * i + lane;
          const int64_t tk = static_cast<int64_t>(w.hk) * T + w.s_doc + rel;
          kw[i] = (rel < w.L ? static_cast<uint32_t>(__ldg(a.k_scales + tk)) : 127u) * 0x01010101u;
          vw[i] = (rel < w.L ? static_cast<uint32_t>(__ldg(a.v_scales + tk)) : 127u) * 0x01010101u;
        }
        reinterpret_cast<uint4*>(smem + Lay::kSfbS)[lane] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
        reinterpret_cast<uint4*>(smem + Lay::kSfbP)[lane] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
      } else {
        // dQ = dS K: K's scale per 32-key group along the contraction
        uint32_t word = 0;
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const int rel = w.kt * kTile + gg * kBlock;
          const uint32_t byte = rel < w.L ? __ldg(a.k_scales + static_cast<int64_t>(w.hk) * T + w.s_doc + rel) : 127u;
          word |= byte << (8 * gg);
        }
        reinterpret_cast<uint4*>(smem + Lay::kSfbDQ)[lane] = make_uint4(word, word, word, word);
      }
      if constexpr (kF4) {
        // the 4-bit S MMA's K scale words: per 64-element chunk c, row r,
        // word i = the four UE4M3 bytes of key row 32 i + r of the tile
        const int64_t k0 = w.s_doc + w.kt * kTile;
#pragma unroll
        for (int c = 0; c < Lay::kC4; ++c) {
          uint32_t wk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t tt = k0 + 32 * i + lane;
            wk[i] = tt < T ? __ldg(reinterpret_cast<const uint32_t*>(a.k4_scales + (tt * a.Hkv + w.hk) * (D / 16)) + c) : 0u;
          }
          reinterpret_cast<uint4*>(smem + Lay::kSk4 + c * 512)[lane] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int32_t y = static_cast<int32_t>(w.s_doc + w.kt * kTile);
        mbar_arrive_expect_tx(&bars[Lay::bKVFull], 2 * Lay::kTileBytes + (kF4 ? Lay::kTileBytes / 2 : 0));
        tma_load_2d(smem + Lay::kK, &a.tm_k, w.hk * D, y, &bars[Lay::bKVFull]);
        tma_load_2d(smem + Lay::kV, &a.tm_v, w.hk * D, y, &bars[Lay::bKVFull]);
        if constexpr (kF4) tma_load_2d(smem + Lay::kK4, &a.tm_k4, w.hk * (D / 2), y, &bars[Lay::bKVFull]);
      }
      __syncwarp();
      ++kv_issued;
      for (int n = 0; n < w.n_it; ++n) {
        int h, qt;
        bwd_iter(w, n, h, qt);
        const int st = it % Lay::kStages;
        if (it >= Lay::kStages &&
            !mbar_wait(&bars[Lay::bQDEmpty + st], ((it / Lay::kStages) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleProducer))) {
          ok = false;
          break;
        }
        // dV = P'^T dO and dK = dS^T Q contract over queries: the dO and Q
        // scale of each 32-query group
        uint32_t wdo = 0, wq = 0;
        if constexpr (kExact) {
          // exact options: dO's and Q's exponents are folded into P' and dS
          wdo = wq = 0x7f7f7f7fu;
        } else {
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            const int rel = qt * kTile + gg * kBlock;
            const int64_t idx = static_cast<int64_t>(h) * T + w.s_doc + rel;
            const uint32_t bdo = rel < w.L ? __ldg(a.do_scales + idx) : 127u;
            const uint32_t bq = rel < w.L ? __ldg(a.q_scales + idx) : 127u;
            wdo |= bdo << (8 * gg);
            wq |= bq << (8 * gg);
          }
        }
        reinterpret_cast<uint4*>(smem + Lay::kSfbDV + st * 512)[lane] = make_uint4(wdo, wdo, wdo, wdo);
        reinterpret_cast<uint4*>(smem + Lay::kSfbDK + st * 512)[lane] = make_uint4(wq, wq, wq, wq);
        if constexpr (kF4) {
          // the 4-bit S MMA's Q scale words of this stage
          const int64_t q0 = w.s_doc + qt * kTile;
#pragma unroll
          for (int c = 0; c < Lay::kC4; ++c) {
            uint32_t wq4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int64_t tt = q0 + 32 * i + lane;
              wq4[i] = tt < T ? __ldg(reinterpret_cast<const uint32_t*>(a.q4_scales + (tt * a.Hq + h) * (D / 16)) + c) : 0u;
            }
            reinterpret_cast<uint4*>(smem + Lay::kSq4 + (st * Lay::kC4 + c) * 512)[lane] =
                make_uint4(wq4[0], wq4[1], wq4[2], wq4[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[Lay::bQDFull + st], 2 * Lay::kTileBytes + (kF4 ? Lay::kTileBytes / 2 : 0));
          const int32_t y = static_cast<int32_t>(w.s_doc + qt * kTile);
          tma_load_2d(smem + Lay::kQ + st * Lay::kTileBytes, &a.tm_q, h * D, y, &bars[Lay::bQDFull + st]);
          tma_load_2d(smem + Lay::kDO + st * Lay::kTileBytes, &a.tm_do, h * D, y, &bars[Lay::bQDFull + st]);
          if constexpr (kF4)
            tma_load_2d(smem + Lay::kQ4 + st * (Lay::kTileBytes / 2), &a.tm_q4, h * (D / 2), y, &bars[Lay::bQDFull + st]);
        }
        __syncwarp();
        ++it;
      }
      if (!ok) break;
      ++items;
      // the next item is claimed once this one's last Q/dO loads are issued
      g = feed.next(rec);
      ok = feed.publish(g, rec);
    }
    if (!ok) *abort_flag = 1;
    // Let every copy still in flight land before the CTA can exit, also when
    // the loop ended because another warp gave up: the last phase armed on
    // each Q/dO stage and on the K/V buffer (already complete after a normal
    // run).
    for (int x = (it > Lay::kStages ? it - Lay::kStages : 0); x < it; ++x)
      mbar_wait(&bars[Lay::bQDFull + (x % Lay::kStages)], (x / Lay::kStages) & 1, nullptr);
    if (kv_issued > 0) mbar_wait(&bars[Lay::bKVFull], (kv_issued - 1) & 1, nullptr);
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      work.whole_warp = false;
      work.sleep = role_sleeps(kSleepMask, kRoleIssuer);
      if constexpr (kExact && !Lay::kFoldCols) {
        // Q and dO enter S and dP with scale 1 (their exponents are in the
        // compute warps' row factors); P''s scales are written per iteration
        uint32_t* sa1 = reinterpret_cast<uint32_t*>(smem + Lay::kSa1);
        for (int i = 0; i < 128; ++i) sa1[i] = 0x7f7f7f7fu;
        fence_proxy_async_smem();
        tmem_cp_32x128b_x4(tbase + Lay::kTSa1, make_smem_desc(smem_u32(sa1), 0, 128, kSwizzleNone));
      } else {
        // P' operand of dV: constant scale 2^-8
        const uint32_t pword = 0x77777777u;  // 119 = 127 - 8 in every byte
        uint32_t* sfa_dv = reinterpret_cast<uint32_t*>(smem + Lay::kSfaDV);
        for (int i = 0; i < 128; ++i) sfa_dv[i] = pword;
        fence_proxy_async_smem();
      }
      const uint32_t idesc_s = idesc_f8(128, 128, false, false);
      const uint32_t sK = smem_u32(smem + Lay::kK);
      const uint32_t sV = smem_u32(smem + Lay::kV);
      const uint32_t sPp = smem_u32(smem + Lay::kPp);
      const uint32_t sDS = smem_u32(smem + Lay::kDS);
      auto sf_desc = [&](int off) { return make_smem_desc(smem_u32(smem + off), 0, 128, kSwizzleNone); };
      int it = 0, items = 0;
      bool ok = true;
      for (;;) {
        int g;
        int4 rec;
        if (!work.next(g, rec) || *abort_flag) break;
        const BwdItem w = decode_bwd(a, g, rec);
        if (!mbar_wait(&bars[Lay::bKVFull], items & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
        if constexpr (kF4 && D == 64) {
          // the item's K scale columns were last read by the previous item's
          // S MMAs, complete before its K/V buffer was released (at d = 128
          // they lie in dP's columns and are copied before every S)
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < Lay::kC4; ++c)
            tmem_cp_32x128b_x4(tbase + Lay::kTSk4 + 4 * c, sf_desc(Lay::kSk4 + c * 512));
        }
        for (int n = 0; n < w.n_it; ++n, ++it) {
          const int st = it % Lay::kStages;
          if (!mbar_wait(&bars[Lay::bQDFull + st], (it / Lay::kStages) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
          if (it > 0) {
            // S/dP columns free: read by the compute warps, the dQ that
            // aliases S drained, and the previous dV and dK MMAs (which read
            // scale factors in dP's columns) complete
            if (!mbar_wait(&bars[Lay::bSdpEmpty], (it - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
            if (!mbar_wait(&bars[Lay::bDqEmpty], (it - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
            if (Lay::kDqFirst && !mbar_wait(&bars[Lay::bDsEmpty], (it - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
          }
          tc_fence_after();
          const uint32_t sQ = smem_u32(smem + Lay::kQ + st * Lay::kTileBytes);
          const uint32_t sDO = smem_u32(smem + Lay::kDO + st * Lay::kTileBytes);
          if constexpr (kF4) {
            // NVFP4 path: S recomputed with the forward's 4-bit MMA (same
            // operands, scales and K order); dP unscaled E4M3.  This stage's
            // Q scale columns were last read by S(it - 2), complete before
            // its Q/dO stage was released.
            constexpr uint32_t kSwz4 = D == 64 ? kSwizzle32B : kSwizzle64B;
            const uint32_t sQ4 = smem_u32(smem + Lay::kQ4 + st * (Lay::kTileBytes / 2));
            const uint32_t sK4 = smem_u32(smem + Lay::kK4);
#pragma unroll
            for (int c = 0; c < Lay::kC4; ++c)
              tmem_cp_32x128b_x4(tbase + Lay::kTSq4 + (st * Lay::kC4 + c) * 4, sf_desc(Lay::kSq4 + (st * Lay::kC4 + c) * 512));
            if constexpr (D == 128) {
              // K's scale columns lie in dP's accumulator, which every dP
              // overwrites: copied again for each S (dP of the previous
              // iteration has been read, so the columns are free)
#pragma unroll
              for (int c = 0; c < Lay::kC4; ++c) tmem_cp_32x128b_x4(tbase + Lay::kTSk4 + 4 * c, sf_desc(Lay::kSk4 + c * 512));
            }
#pragma unroll
            for (int c = 0; c < Lay::kC4; ++c) {
              mma_mxf4nvf4(tbase + Lay::kTS, make_smem_desc(sQ4 + 32 * c, 16, 8 * (D / 2), kSwz4),
                           make_smem_desc(sK4 + 32 * c, 16, 8 * (D / 2), kSwz4), idesc_mxf4nvf4(128, 128),
                           tbase + Lay::kTSq4 + (st * Lay::kC4 + c) * 4, tbase + Lay::kTSk4 + 4 * c, c > 0 ? 1u : 0u);
            }
            if constexpr (D == 128) {
              // the scale columns sit inside dP's accumulator: S completes first
              mma_commit(&bars[Lay::bSDone]);
              if (!mbar_wait(&bars[Lay::bSDone], it & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              mma_f8(tbase + Lay::kTdP, make_smem_desc(sDO + 32 * kk, 16, 8 * D, Lay::kSwz),
                     make_smem_desc(sV + 32 * kk, 16, 8 * D, Lay::kSwz), idesc_s, kk > 0 ? 1u : 0u);
            }
          } else if constexpr (kExact && !Lay::kFoldCols) {
            // per-key K and V scales (exact options): block-scaled S and dP.
            // The columns were last read by S/dP of the previous iteration,
            // complete since the compute warps released it.
            tmem_cp_32x128b_x4(tbase + Lay::kTSbS, sf_desc(Lay::kSfbS));
            tmem_cp_32x128b_x4(tbase + Lay::kTSbP, sf_desc(Lay::kSfbP));
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              mma_mxf8(tbase + Lay::kTS, make_smem_desc(sQ + 32 * kk, 16, 8 * D, Lay::kSwz),
                       make_smem_desc(sK + 32 * kk, 16, 8 * D, Lay::kSwz), idesc_mxf8(128, 128, false, false, kk, kk),
                       tbase + Lay::kTSa1, tbase + Lay::kTSbS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              mma_mxf8(tbase + Lay::kTdP, make_smem_desc(sDO + 32 * kk, 16, 8 * D, Lay::kSwz),
                       make_smem_desc(sV + 32 * kk, 16, 8 * D, Lay::kSwz), idesc_mxf8(128, 128, false, false, kk, kk),
                       tbase + Lay::kTSa1, tbase + Lay::kTSbP, kk > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              mma_f8(tbase + Lay::kTS, make_smem_desc(sQ + 32 * kk, 16, 8 * D, Lay::kSwz),
                     make_smem_desc(sK + 32 * kk, 16, 8 * D, Lay::kSwz), idesc_s, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              mma_f8(tbase + Lay::kTdP, make_smem_desc(sDO + 32 * kk, 16, 8 * D, Lay::kSwz),
                     make_smem_desc(sV + 32 * kk, 16, 8 * D, Lay::kSwz), idesc_s, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&bars[Lay::bSdpFull]);
          if (!mbar_wait(&bars[Lay::bDsFull], it & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
          if (D == 64 && it > 0 && !mbar_wait(&bars[Lay::bDqEmpty], (it - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
          if (n == 0 && items > 0 && !mbar_wait(&bars[Lay::bAccEmpty], (items - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) {
            ok = false;
            break;
          }
          tc_fence_after();
          tmem_cp_32x128b_x4(tbase + Lay::kTSfaDV, sf_desc(Lay::kSfaDV));
          tmem_cp_32x128b_x4(tbase + Lay::kTSfbDV, sf_desc(Lay::kSfbDV + st * 512));
          tmem_cp_32x128b_x4(tbase + Lay::kTSfaDK, sf_desc(Lay::kSfaDK));
          tmem_cp_32x128b_x4(tbase + Lay::kTSfbDK, sf_desc(Lay::kSfbDK + st * 512));
          tmem_cp_32x128b_x4(tbase + Lay::kTSfaDQ, sf_desc(Lay::kSfaDQ));
          tmem_cp_32x128b_x4(tbase + Lay::kTSfbDQ, sf_desc(Lay::kSfbDQ));
          const uint32_t acc_on = (n > 0) ? 1u : 0u;
          // dQ = dS K   (A: dS K-major, B: K MN-major); the exact options'
          // dQ payload has its own tile
          const uint32_t sDSq = kExact ? smem_u32(smem + Lay::kDS2) : sDS;
          auto issue_dq = [&]() {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              mma_mxf8(tbase + Lay::kTdQ, make_smem_desc(sDSq + 32 * kk, 16, 1024, kSwizzle128B),
                       make_smem_desc(sK + kk * 32 * D, 16, 8 * D, Lay::kSwz), idesc_mxf8(128, D, false, true, kk, kk),
                       tbase + Lay::kTSfaDQ, tbase + Lay::kTSfbDQ, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars[Lay::bDqFull]);
          };
          if constexpr (Lay::kDqFirst) issue_dq();
          // dV += P'^T dO   (A: P' viewed MN-major, B: dO MN-major)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_mxf8(tbase + Lay::kTdV, make_smem_desc(sPp + kk * 4096, 16, 1024, kSwizzle128B),
                     make_smem_desc(sDO + kk * 32 * D, 16, 8 * D, Lay::kSwz), idesc_mxf8(128, D, true, true, kk, kk),
                     tbase + Lay::kTSfaDV, tbase + Lay::kTSfbDV, (acc_on || kk > 0) ? 1u : 0u);
          }
          // dK += dS^T Q
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_mxf8(tbase + Lay::kTdK, make_smem_desc(sDS + kk * 4096, 16, 1024, kSwizzle128B),
                     make_smem_desc(sQ + kk * 32 * D, 16, 8 * D, Lay::kSwz), idesc_mxf8(128, D, true, true, kk, kk),
                     tbase + Lay::kTSfaDK, tbase + Lay::kTSfbDK, (acc_on || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars[Lay::bDsEmpty]);
          mma_commit(&bars[Lay::bQDEmpty + st]);
          if constexpr (!Lay::kDqFirst) issue_dq();

        }
        if (!ok) break;
        mma_commit(&bars[Lay::bKVEmpty]);
        ++items;
      }
      if (!ok) *abort_flag = 1;
      mma_commit(&bars[Lay::bFinal]);
      mbar_wait(&bars[Lay::bFinal], 0, nullptr);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == Lay::kWMma) tmem_dealloc(tbase, 512);
}

template <int D, bool kExact, bool kDump = false, bool kF4 = false>
static void launch_bwd_t(const BwdArgs& a, int num_ctas, cudaStream_t st) {
  constexpr int smem = BwdLayout<D, kExact, kF4>::kSmemAlloc;
  static std::atomic<uint64_t> configured{0};
  if (first_use_on_device(configured))
    cudaFuncSetAttribute(bwd_kernel<D, kExact, kDump, kF4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  bwd_kernel<D, kExact, kDump, kF4><<<num_ctas, BwdLayout<D, kExact, kF4>::kThreads, smem, st>>>(a);
}

// d = 64 runs bwd64_kernel, except for the exact options (this kernel with
// the exact variant; TMEM has no room for the S/dP scale factors at d = 128)
cudaError_t launch_bwd(const BwdArgs& a, int d, int num_ctas, cudaStream_t st) {
  if (a.nvfp4) {
    // the NVFP4 path: the eight-score-warp kernel at d = 64, this one at 128
    if (a.exact || a.dump.s != nullptr) return cudaErrorInvalidValue;
    if (d == 64) return launch_bwd_d64(a, num_ctas, st);
    launch_bwd_t<128, false, false, true>(a, num_ctas, st);
    return cudaGetLastError();
  }
  if (a.exact && d == 128 && a.dump.s == nullptr) {
    launch_bwd_t<128, true>(a, num_ctas, st);
    return cudaGetLastError();
  }
  if (a.dump.s != nullptr) {
    // diagnostic score-tile dump (token-block scales only)
    if (a.exact) return cudaErrorInvalidValue;
    if (d == 64) return launch_bwd_d64(a, num_ctas, st);
    launch_bwd_t<128, false, true>(a, num_ctas, st);
    return cudaGetLastError();
  }
  // d = 64, with or without the exact options: the eight-score-warp kernel
  if (d == 64) return launch_bwd_d64(a, num_ctas, st);
  launch_bwd_t<128, false>(a, num_ctas, st);
  return cudaGetLastError();
}

}  // namespace flamia
