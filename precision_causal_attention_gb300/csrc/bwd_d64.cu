// MXFP8 causal packed attention backward at head dimension 64, sm_103a.
//
// Method: FLAMIA (arXiv 2611.03344) Sections 2, 3.1, 3.3, 3.5.3 and
// Appendix B.1; the arithmetic of every tile is that of the general backward
// kernel (S recomputed bitwise as in the forward, P = 2^(S2 - LSE2),
// dS = P o (dP - D) quantized per 32x32 block with the round-up exponent,
// P' = E4M3(2^8 P) with scale 2^-8, block-scaled MMAs for dV, dK, dQ).  What
// differs is the schedule.  One iteration n is one query tile of one query
// head against the CTA's key tile; the MMA warps issue, per iteration,
//     S(n+1), dP(n+1)            as soon as the compute warps have read S/dP(n)
//     dQ(n) = dS(n) K            once dS(n) is in shared memory
//     dV += P'(n)^T dO(n),  dK += dS(n)^T Q(n)
// and a separate warpgroup drains dQ(n) to the fp32 accumulator and writes
// dV/dK at the end of an item, so the score warps do nothing but score work.
// The P' and dS tiles, their block-scale words and the scale-factor columns
// in tensor memory are double-buffered by the parity of n.  The iteration
// stream runs across work items: K/V are double-buffered per item and the
// first S/dP of the next item is issued during the last iteration of the
// current one.
//
// Warp roles (512 threads, one CTA per SM, 512 TMEM columns; registers are
// moved between warpgroups with setmaxnreg):
//   warps 0-7   score warps (160 registers).  Warp w reads TMEM lanes
//               32(w%4)..+31 (query rows); warpgroup c = w/4 takes score
//               columns [64c, 64c+64).
//   warps 8-11  dQ / epilogue warps (112 registers): lanes 32(w%4)..+31 of dQ
//               (query rows) each iteration, and of dV, dK (key rows) at the
//               end of an item; one TMA reduce-add per warp and 32 columns.
//   warp 12     TMA producer: K/V per item (2 buffers), Q/dO per iteration
//               (5-stage ring; 3 stages for the variants below), and the
//               scale words derived from token scales
//   warp 13     MMA issuer for S/dP (lane 0) and TMEM owner
//   warp 14     MMA issuer for dV and dK (lane 0)
//   warp 15     MMA issuer for dQ (lane 0); warps 12-15 run with 80 registers
// TMEM: S [0,128) dP [128,256) dV [256,320) dK [320,384) dQ [384,448)
//       scale factors [448,492): the constant P' scale, K's scales per K/V
//       buffer, and two per-iteration sets (dS for dQ and dK, dO, Q).
//
// Variants (template flags):
//   kDet    dQ partials as 64-bit fixed-point integers, added per query row
//           with integer bulk reduce-adds (order-independent sums).
//   kExact  the exact options (Section 3.2, Appendix A.3): S and dP take K's
//           and V's per-key exponents as exact column factors from a
//           per-warp fold table, P' carries dO's per-token exponent relative
//           to its 32-query block (per-parity scale words, TMEM up to 500),
//           dK's payload Q's, and dQ reads its own K-folded payload tile with
//           per-row exponents.
//   kF4     the mixed NVFP4/FP8 path (Section 3.4): S is recomputed with one
//           kind::mxf4nvf4 MMA from E2M1 Q and K tiles (their UE4M3 scale
//           columns at [492,512)); dP and the rest stay E4M3.
#include <cuda_bf16.h>
#include <cstdint>

#include "bwd_common.cuh"

namespace flamia {

template <bool kExact = false, bool kF4 = false>
struct Bwd64LayoutT {
  static constexpr int D = 64;
  // the exact options keep a second dS tile (the dQ payload) and per-warp
  // fold tables in shared memory, the NVFP4 path the 4-bit Q and K tiles of
  // the recomputed S with their scale words: their Q/dO ring has 3 stages
  static constexpr int kStages = (kExact || kF4) ? 3 : 5;
  static constexpr int kTileBytes = kTile * D;                // 8 KB of E4M3 codes
  static constexpr int kPTileBytes = kTile * kTile;           // 16 KB
  static constexpr uint32_t kSwz = kSwizzle64B;
  // shared memory (every tile offset a multiple of 1024 B)
  static constexpr int kK = 0;                                // 2 buffers
  static constexpr int kV = kK + 2 * kTileBytes;              // 2 buffers
  static constexpr int kQ = kV + 2 * kTileBytes;              // kStages tiles
  static constexpr int kDO = kQ + kStages * kTileBytes;       // kStages tiles
  static constexpr int kPp = kDO + kStages * kTileBytes;      // 2 x P' codes [128 q][128 k], 128B swizzle
  static constexpr int kDS = kPp + 2 * kPTileBytes;           // 2 x dS codes [128 q][128 k]
  // dQ staging for the bulk reduce-add, kDqWarpBytes per drain warp: two
  // boxes of 32 rows x 32 fp32 (128B swizzle), box (quad, half) at
  // kDQs + quad * kDqWarpBytes + half * kDqBoxBytes.  The deterministic
  // option uses the same area as one slot of 32 rows x kDetRowBytes (32
  // fixed-point columns per row, padded so the rows start in different banks).
  static constexpr int kDqBoxBytes = 32 * 128;
  static constexpr int kDetRowBytes = 272;
  static constexpr int kDetSlotBytes = 32 * kDetRowBytes;
  static constexpr int kDqWarpBytes = 9 * 1024;
  static constexpr int kDQs = kDS + 2 * kPTileBytes;
  // scale words, [32 rows][16 B] each, laid out for tcgen05.cp 32x128b
  static constexpr int kSfaDV = kDQs + 4 * kDqWarpBytes;      // constant 2^-8 (exact options: per parity)
  static constexpr int kSfaDQ = kSfaDV + (kExact ? 2 : 1) * 512;   // per parity
  static constexpr int kSfaDK = kSfaDQ + 2 * 512;             // per parity
  static constexpr int kSfbDQ = kSfaDK + 2 * 512;             // per K/V buffer
  static constexpr int kSfbDV = kSfbDQ + 2 * 512;             // per stage
  static constexpr int kSfbDK = kSfbDV + kStages * 512;       // per stage
  // exact options: the dQ payload tile per parity (dS times K's per-key
  // factors, per-row exponents), and per score warp the fold table of its 64
  // keys: K's and V's factors 2^(E(j) - G_g) and each 32-key group's largest
  // scale byte G_g (two for K, two for V)
  static constexpr int kDS2 = (kSfbDK + kStages * 512 + 1023) / 1024 * 1024;
  static constexpr int kFoldBytes = 2 * 64 * 4 + 16;
  static constexpr int kFold = kDS2 + 2 * kPTileBytes;
  // NVFP4 path: the E2M1 Q tile of each stage and K tile of each K/V buffer
  // (128 rows x 32 bytes, 32B swizzle) and the 4-bit S MMA's scale words (Q
  // per stage, K per K/V buffer)
  static constexpr int kTile4Bytes = kTile * D / 2;
  static constexpr int kQ4 = (kSfbDK + kStages * 512 + 1023) / 1024 * 1024;
  static constexpr int kK4 = kQ4 + kStages * kTile4Bytes;
  static constexpr int kSq4 = kK4 + 2 * kTile4Bytes;
  static constexpr int kSk4 = kSq4 + kStages * 512;
  static constexpr int kBar = kExact ? kFold + 8 * kFoldBytes : (kF4 ? kSk4 + 2 * 512 : kSfbDK + kStages * 512);
  enum {
    bKVFull = 0,
    bKVEmpty = bKVFull + 2,
    bQDFull = bKVEmpty + 2,
    bQDEmpty = bQDFull + kStages,
    bSdpFull = bQDEmpty + kStages,
    bSdpEmpty,
    // 2, per parity of the iteration: a score warp can run one iteration
    // ahead of the slowest (S/dP(it+1) is issued once every warp has read
    // S/dP(it)), so its ds_full(it+1) arrival must not land on the phase
    // that still collects ds_full(it)
    bDsFull,
    bDsEmpty = bDsFull + 2,     // 2, per parity
    bDqFull = bDsEmpty + 2,
    bDqEmpty,
    bAccFull,
    bAccEmpty,
    bFinal,
    bFinal2,
    bFinal3,
    kNumBars
  };
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 8;
  static constexpr int kRing = (kAbort + 16 + 15) / 16 * 16;   // work hand-out ring (ItemRing)
  static constexpr int kBytes = kRing + static_cast<int>(sizeof(ItemRing));
  static constexpr int kSmemAlloc = kBytes + 1024;
  static constexpr int kComputeThreads = 256;
  static constexpr int kDrainThreads = 128;
  static constexpr int kThreads = 512;
  static constexpr uint32_t kRegsCompute = 160, kRegsDrain = 112, kRegsService = 80;
  // tensor memory columns
  static constexpr uint32_t kTS = 0;
  static constexpr uint32_t kTdP = 128;
  static constexpr uint32_t kTdV = 256;
  static constexpr uint32_t kTdK = 320;
  static constexpr uint32_t kTdQ = 384;
  static constexpr uint32_t kTSfaDV = 448;                    // constant
  static constexpr uint32_t kTSfbDQ = 452;                    // + 4 x K/V buffer
  static constexpr uint32_t kTSet = 460;                      // + kSetCols x parity
  static constexpr uint32_t kSfaDQo = 0, kSfbDVo = 4, kSfaDKo = 8, kSfbDKo = 12;
  // exact options: P''s scale per 32-query block (dV's A operand) per parity
  static constexpr uint32_t kSfaDVo = 16;
  static constexpr uint32_t kSetCols = kExact ? 20 : 16;
  // NVFP4 path: the 4-bit S MMA's scale columns, Q per stage and K per K/V buffer
  static constexpr uint32_t kTSq4 = kTSet + 2 * kSetCols;
  static constexpr uint32_t kTSk4 = kTSq4 + 4 * kStages;
  static constexpr float kSmScale = 0.18033688011112042f;     // log2(e) / sqrt(64)
  static constexpr float kInvSqrtD = 0.125f;
};
using Bwd64Layout = Bwd64LayoutT<false>;
static_assert(Bwd64Layout::kSmemAlloc <= 227 * 1024, "shared memory budget");
static_assert(Bwd64LayoutT<true>::kSmemAlloc <= 227 * 1024, "shared memory budget (exact options)");
static_assert(Bwd64Layout::kTSet + 2 * Bwd64Layout::kSetCols <= 512, "tensor memory budget");
static_assert(Bwd64LayoutT<true>::kTSet + 2 * Bwd64LayoutT<true>::kSetCols <= 512, "tensor memory budget (exact options)");
static_assert(Bwd64LayoutT<true>::kDS2 % 1024 == 0 && Bwd64LayoutT<true>::kFold % 16 == 0, "exact options layout");
static_assert(Bwd64LayoutT<false, true>::kSmemAlloc <= 227 * 1024, "shared memory budget (NVFP4 path)");
static_assert(Bwd64LayoutT<false, true>::kTSk4 + 8 <= 512, "tensor memory budget (NVFP4 path)");
static_assert(Bwd64LayoutT<false, true>::kQ4 % 1024 == 0 && Bwd64LayoutT<false, true>::kK4 % 1024 == 0,
              "4-bit tiles need 1024 B alignment");
static_assert(Bwd64Layout::kDQs % 1024 == 0 && Bwd64Layout::kPp % 1024 == 0 && Bwd64Layout::kDqWarpBytes % 1024 == 0,
              "swizzled tiles need 1024 B alignment");
static_assert(2 * Bwd64Layout::kDqBoxBytes <= Bwd64Layout::kDqWarpBytes &&
                  Bwd64Layout::kDetSlotBytes <= Bwd64Layout::kDqWarpBytes,
              "dQ staging per drain warp");
// the launch gives every thread 65536 / 512 = 128 registers; the warpgroups'
// shares after setmaxnreg must fit in that pool (and in each SMSP's quarter,
// which holds one warp of every warpgroup)
static_assert((2 * Bwd64Layout::kRegsCompute + Bwd64Layout::kRegsDrain + Bwd64Layout::kRegsService) * 128 <= 65536,
              "register split exceeds the launch allocation");

template <bool kDump = false, bool kDet = false, bool kExact = false, bool kF4 = false>
__global__ void __launch_bounds__(Bwd64Layout::kThreads, 1) bwd64_kernel(const __grid_constant__ BwdArgs a) {
  using Lay = Bwd64LayoutT<kExact, kF4>;
  // the producer sleeps in its waits (it runs well ahead of the MMAs); the
  // other roles poll (sleeping changed the backward's time by under 1 %)
  constexpr unsigned kSleepMask = kRoleProducer;
  static_assert(!(kExact && kF4), "the NVFP4 path and the exact options are separate");
  constexpr int D = Lay::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Lay::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[Lay::bKVFull + s], 1);
      mbar_init(&bars[Lay::bKVEmpty + s], 2);      // S/dP issuer and dQ issuer
      mbar_init(&bars[Lay::bDsEmpty + s], 2);      // one commit from each MMA issuer
    }
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&bars[Lay::bQDFull + s], 1);
      mbar_init(&bars[Lay::bQDEmpty + s], 1);
    }
    mbar_init(&bars[Lay::bSdpFull], 1);
    mbar_init(&bars[Lay::bSdpEmpty], Lay::kComputeThreads);
    mbar_init(&bars[Lay::bDsFull], Lay::kComputeThreads);
    mbar_init(&bars[Lay::bDsFull + 1], Lay::kComputeThreads);
    mbar_init(&bars[Lay::bDqFull], 1);
    mbar_init(&bars[Lay::bDqEmpty], Lay::kDrainThreads);
    mbar_init(&bars[Lay::bAccFull], 1);
    mbar_init(&bars[Lay::bAccEmpty], Lay::kDrainThreads);
    mbar_init(&bars[Lay::bFinal], 1);
    mbar_init(&bars[Lay::bFinal2], 1);
    mbar_init(&bars[Lay::bFinal3], 1);
    // consumers of the item ring: 8 score warps, 4 dQ warps, 3 MMA issuers
    reinterpret_cast<ItemRing*>(smem + Lay::kRing)->init(15);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 13) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (warp == 12 && lane == 0) {
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

  if (warp < 8) {
    // ------------------------------------------------------------ score warps
    setmaxnreg_inc<Lay::kRegsCompute>();
    work.sleep = role_sleeps(kSleepMask, kRoleCompute);
    const int quad = warp & 3, wg = warp >> 2;
    const int row = quad * 32 + lane;                 // TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
    const uint32_t rbase = (row >> 3) * 1024 + (row & 7) * 128;
    int it = 0;
    bool ok = true;
    for (;;) {
      int g;
      int4 rec;
      if (!work.next(g, rec) || *abort_flag) break;
      const BwdItem w = decode_bwd(a, g, rec);
      // scales of this warpgroup's two 32-key groups
      int ek0, ek1, ev0, ev1;
      {
        const int rel = w.kt * kTile + 2 * wg * kBlock;
        const int64_t tk = static_cast<int64_t>(w.hk) * T + w.s_doc + rel;
        ek0 = rel < w.L ? static_cast<int>(__ldg(a.k_scales + tk)) - 127 : 0;
        ev0 = rel < w.L ? static_cast<int>(__ldg(a.v_scales + tk)) - 127 : 0;
        ek1 = rel + kBlock < w.L ? static_cast<int>(__ldg(a.k_scales + tk + kBlock)) - 127 : 0;
        ev1 = rel + kBlock < w.L ? static_cast<int>(__ldg(a.v_scales + tk + kBlock)) - 127 : 0;
      }
      // exact options: this warp's fold table of its 64 keys, rewritten per
      // item (the warp is past its previous item's iterations).  Per key j
      // the factors 2^(E_K(j) - G_g) and 2^(E_V(j) - Gv_g), with G_g and
      // Gv_g the 32-key group's largest K and V scale bytes; keys past the
      // document end get factor 0.  S and dP take them as column factors
      // (the products are exact, so S2 and dP round as with the scales inside
      // the MMA), and dQ's payload takes K's.
      float* fold = reinterpret_cast<float*>(smem + (kExact ? Lay::kFold + warp * Lay::kFoldBytes : 0));
      if constexpr (kExact) {
        int* gmaxs = reinterpret_cast<int*>(fold + 128);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int kj = w.kt * kTile + 64 * wg + 32 * jj + lane;
          const int64_t tk = static_cast<int64_t>(w.hk) * T + w.s_doc + kj;
          const int kbyte = kj < w.L ? static_cast<int>(__ldg(a.k_scales + tk)) : -1;
          const int vbyte = kj < w.L ? static_cast<int>(__ldg(a.v_scales + tk)) : -1;
          const int gk = max(__reduce_max_sync(0xffffffffu, kbyte), 0);
          const int gv = max(__reduce_max_sync(0xffffffffu, vbyte), 0);
          fold[32 * jj + lane] = kbyte >= 0 ? pow2_any(kbyte - gk) : 0.f;
          fold[64 + 32 * jj + lane] = vbyte >= 0 ? pow2_any(vbyte - gv) : 0.f;
          if (lane == 0) {
            gmaxs[jj] = gk;
            gmaxs[2 + jj] = gv;
          }
        }
        __syncwarp();
      }
      // per-row scalars of the next iteration, loaded one iteration ahead and
      // converted only when used
      struct RowVals { uint32_t eqb, edob; float lse, Di; };
      auto load_row = [&](const BwdCursor& c) {
        RowVals v;
        const int qi = min(c.qt * kTile + row, w.L - 1);
        const int64_t ht = static_cast<int64_t>(c.h) * T + w.s_doc + qi;
        v.eqb = __ldg(a.q_scales + ht);
        v.edob = __ldg(a.do_scales + ht);
        v.lse = __ldg(a.lse + ht);
        v.Di = __ldg(a.D + ht);
        return v;
      };
      BwdCursor cur, nxt;
      cur.begin(w);
      nxt = cur;
      RowVals rv_next = load_row(cur);
      for (int n = 0; n < w.n_it; ++n, ++it) {
        const int qt = cur.qt;
        const RowVals rv = rv_next;
        if (n + 1 < w.n_it) {
          nxt.advance(w);
          rv_next = load_row(nxt);
        }
        const int qi = qt * kTile + row;
        const bool valid = qi < w.L;
        // A row past the document end is zeroed through its exponent offset
        // (arg_add = -inf gives P = 0, P' = 0 and dS = 0 in every column), so
        // it needs no column mask.
        int nvis;
        if (!valid) nvis = kTile;
        else if (a.causal) nvis = (qt == w.kt) ? row + 1 : kTile;
        else nvis = min(kTile, w.L - w.kt * kTile);
        const bool full = __all_sync(0xffffffffu, nvis >= 64 * wg + 64);
        // 2^8 P = 2^(S2 - LSE2 + 8) is the dV operand directly; dS is carried
        // as 2^8 dS, the factor leaving the block exponent exactly
        const float arg_add = valid ? 8.f - rv.lse * kLog2e : -INFINITY;
        const int r_eq = valid ? static_cast<int>(rv.eqb) - 127 : 0;
        const int r_edo = valid ? static_cast<int>(rv.edob) - 127 : 0;
        const float negD = valid ? -rv.Di : 0.f;
        const int pb = it & 1;

        if (!mbar_wait(&bars[Lay::bSdpFull], it & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
        // the MMAs of iteration it-2 are done with this parity's P'/dS tiles and scale words
        if (it >= 2 && !mbar_wait(&bars[Lay::bDsEmpty + pb], ((it >> 1) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
        tc_fence_after();
        uint8_t* sPp = smem + Lay::kPp + pb * Lay::kPTileBytes;
        uint8_t* sDS = smem + Lay::kDS + pb * Lay::kPTileBytes;
        // exact options: dV's operand E4M3(2^8 P 2^(E_dO(i) - H_b)) carries
        // the row's dO exponent relative to sigma_b = max(H_b - 8, -127), H_b
        // the largest dO exponent among the document rows of this warp's
        // 32-query block; sigma_b is the block's scale along the dV
        // contraction (one byte per block, written by warpgroup 0)
        float fo = 1.f;
        if constexpr (kExact) {
          const int hb = __reduce_max_sync(0xffffffffu, valid ? r_edo : -100000);
          const int sig = max(hb - 8, -127);
          if (valid) fo = pow2_any(r_edo - sig - 8);
          if (wg == 0) {
            uint8_t* dv_bytes = smem + Lay::kSfaDV + pb * 512;
#pragma unroll
            for (int i = 0; i < 4; ++i) dv_bytes[(lane * 4 + i) * 4 + quad] = static_cast<uint8_t>(sig + 127);
          }
        }
        // The two 32-key groups run through one copy of the loop body (not
        // unrolled): the score code stays small enough for the instruction
        // cache it shares with the MMA, producer and dQ warps.
        int Eds0 = 0, Eds1 = 0, Edq0 = 0, Edq1 = 0;
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
          const int gg = 2 * wg + j;
          uint32_t sa[32], pa[32];
          tmem_ld32x2_sync(tbase + lane_base + Lay::kTS + 32 * gg, sa, tbase + lane_base + Lay::kTdP + 32 * gg, pa);
          if (j == 1) {
            // S/dP(it) fully read: the MMA warp may overwrite them with S/dP(it+1)
            tc_fence_before();
            mbar_arrive(&bars[Lay::bSdpEmpty]);
          }
          int gke = j ? ek1 : ek0, gve = j ? ev1 : ev0;
          if constexpr (kExact) {
            const float4* fk4 = reinterpret_cast<const float4*>(fold + 32 * j);
            const float4* fv4 = reinterpret_cast<const float4*>(fold + 64 + 32 * j);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 fk = fk4[u], fv = fv4[u];
              float x0, x1, x2, x3;
              fmul2(x0, x1, __uint_as_float(sa[4 * u]), __uint_as_float(sa[4 * u + 1]), fk.x, fk.y);
              fmul2(x2, x3, __uint_as_float(sa[4 * u + 2]), __uint_as_float(sa[4 * u + 3]), fk.z, fk.w);
              sa[4 * u] = __float_as_uint(x0); sa[4 * u + 1] = __float_as_uint(x1);
              sa[4 * u + 2] = __float_as_uint(x2); sa[4 * u + 3] = __float_as_uint(x3);
              fmul2(x0, x1, __uint_as_float(pa[4 * u]), __uint_as_float(pa[4 * u + 1]), fv.x, fv.y);
              fmul2(x2, x3, __uint_as_float(pa[4 * u + 2]), __uint_as_float(pa[4 * u + 3]), fv.z, fv.w);
              pa[4 * u] = __float_as_uint(x0); pa[4 * u + 1] = __float_as_uint(x1);
              pa[4 * u + 2] = __float_as_uint(x2); pa[4 * u + 3] = __float_as_uint(x3);
            }
            const int* gmaxs = reinterpret_cast<const int*>(fold + 128);
            gke = gmaxs[j] - 127;
            gve = gmaxs[2 + j] - 127;
          }
          // (the NVFP4 path's Q and K scales are inside the S MMA)
          const float cg = kF4 ? Lay::kSmScale : scale_pow2(Lay::kSmScale, r_eq + gke);
          const float cdp = scale_pow2(1.f, r_edo + gve);
          if constexpr (kDump) {
            // diagnostic copy of the recomputed raw S tile and the group factors
            if (w.doc == a.dump.doc && w.kt == a.dump.kt && cur.h == a.dump.h && qt == a.dump.qt) {
#pragma unroll
              for (int c = 0; c < 32; ++c) a.dump.s[row * kTile + 32 * gg + c] = __uint_as_float(sa[c]);
              a.dump.f[row * 4 + gg] = cg;
            }
          }
          // masked scores (beyond the causal diagonal or the document end)
          // become -inf, whose exponential is an exact 0: P' = 0 and dS = 0
          // there, through the same code as fully visible tiles
          if (!full) {
            const int vis = nvis - 32 * gg;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c >= vis) sa[c] = 0xff800000u;
          }
          float ds[32];
          uint32_t pw[8];
          float amax = 0.f, amax2 = 0.f;     // two chains, joined below
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            float a0, a1, a2, a3, t0, t1, t2, t3;
            ffma2(a0, a1, __uint_as_float(sa[c]), __uint_as_float(sa[c + 1]), cg, cg, arg_add, arg_add);
            ffma2(a2, a3, __uint_as_float(sa[c + 2]), __uint_as_float(sa[c + 3]), cg, cg, arg_add, arg_add);
            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1), p2 = ex2_approx(a2), p3 = ex2_approx(a3);
            ffma2(t0, t1, __uint_as_float(pa[c]), __uint_as_float(pa[c + 1]), cdp, cdp, negD, negD);
            ffma2(t2, t3, __uint_as_float(pa[c + 2]), __uint_as_float(pa[c + 3]), cdp, cdp, negD, negD);
            fmul2(ds[c], ds[c + 1], p0, p1, t0, t1);
            fmul2(ds[c + 2], ds[c + 3], p2, p3, t2, t3);
            amax = max3f(amax, fabsf(ds[c]), fabsf(ds[c + 1]));
            amax2 = max3f(amax2, fabsf(ds[c + 2]), fabsf(ds[c + 3]));
            if constexpr (kExact) {
              float q0, q1, q2, q3;
              fmul2(q0, q1, p0, p1, fo, fo);
              fmul2(q2, q3, p2, p3, fo, fo);
              pw[c >> 2] = cvt_e4m3x4(q0, q1, q2, q3);
            } else {
              pw[c >> 2] = cvt_e4m3x4(p0, p1, p2, p3);
            }
          }
          // 32x32 block of dS: this warp's 32 query rows x these 32 keys.  The
          // exponent of 2^8 dS is 8 more than that of dS (clamped at -127).
          amax = fmaxf(amax, amax2);
          float inv;
          if constexpr (kExact) {
            // dK payload: y = dS 2^E_Q(i) = ds 2^(E_Q(i) - 8) in 32x32 blocks
            const int et = amax > 0.f ? roundup_exponent_unclamped(__float_as_uint(amax)) + r_eq - 8 : -100000;
            const int E = min(max(__reduce_max_sync(0xffffffffu, et), -127), 127);
            if (j) Eds1 = E; else Eds0 = E;
            inv = pow2_any(r_eq - 8 - E);
          } else {
            const int E8 = roundup_exponent_from_bits(warp_max_u32(__float_as_uint(amax)));
            const int E = E8 - 8 < -127 ? -127 : E8 - 8;
            if (j) Eds1 = E; else Eds0 = E;
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
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int k = 2 * gg + hf;
            const uint32_t off = rbase + ((k ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(sPp + off) = make_uint4(pw[4 * hf], pw[4 * hf + 1], pw[4 * hf + 2], pw[4 * hf + 3]);
            *reinterpret_cast<uint4*>(sDS + off) = make_uint4(dw[4 * hf], dw[4 * hf + 1], dw[4 * hf + 2], dw[4 * hf + 3]);
          }
          if constexpr (kExact) {
            // dQ payload (K fold, one exponent per query row and 32-key
            // group): x = dS 2^E_K(j), computed as x' = ds 2^(E_K(j) - G_g),
            // so x = x' 2^(G_g - 135) with G_g the group's largest K byte
            const float4* fk4 = reinterpret_cast<const float4*>(fold + 32 * j);
            float ax = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float4 f = fk4[u];
              fmul2(ds[4 * u], ds[4 * u + 1], ds[4 * u], ds[4 * u + 1], f.x, f.y);
              fmul2(ds[4 * u + 2], ds[4 * u + 3], ds[4 * u + 2], ds[4 * u + 3], f.z, f.w);
              ax = max3f(ax, fabsf(ds[4 * u]), fabsf(ds[4 * u + 1]));
              ax = max3f(ax, fabsf(ds[4 * u + 2]), fabsf(ds[4 * u + 3]));
            }
            const int gk = reinterpret_cast<const int*>(fold + 128)[j];
            const int eq_ = ax > 0.f ? roundup_exponent_unclamped(__float_as_uint(ax)) + gk - 135 : -127;
            const int Eq = min(max(eq_, -127), 127);
            if (j) Edq1 = Eq; else Edq0 = Eq;
            const float invq = pow2_any(gk - 135 - Eq);
            uint32_t qw[8];
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              float s0, s1, s2, s3;
              fmul2(s0, s1, ds[c], ds[c + 1], invq, invq);
              fmul2(s2, s3, ds[c + 2], ds[c + 3], invq, invq);
              qw[c >> 2] = cvt_e4m3x4(s0, s1, s2, s3);
            }
            uint8_t* sDS2 = smem + Lay::kDS2 + pb * Lay::kPTileBytes;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int k = 2 * gg + hf;
              const uint32_t off = rbase + ((k ^ (row & 7)) << 4);
              *reinterpret_cast<uint4*>(sDS2 + off) = make_uint4(qw[4 * hf], qw[4 * hf + 1], qw[4 * hf + 2], qw[4 * hf + 3]);
            }
          }
        }
        // block-scale bytes of dS.  dQ = dS K contracts over keys: query row
        // 32 quad + r reads byte gg = E(quad, gg).  dK = dS^T Q contracts over
        // queries: key row 32 gg + r reads byte quad = E(quad, gg).
        {
          // exact options: dQ's payload has its own per-row exponents
          const int q0e = kExact ? Edq0 : Eds0, q1e = kExact ? Edq1 : Eds1;
          const uint32_t half = static_cast<uint32_t>(q0e + 127) | (static_cast<uint32_t>(q1e + 127) << 8);
          reinterpret_cast<uint16_t*>(smem + Lay::kSfaDQ + pb * 512)[(lane * 4 + quad) * 2 + wg] =
              static_cast<uint16_t>(half);
          uint8_t* dk_bytes = smem + Lay::kSfaDK + pb * 512;
          dk_bytes[(lane * 4 + 2 * wg) * 4 + quad] = static_cast<uint8_t>(Eds0 + 127);
          dk_bytes[(lane * 4 + 2 * wg + 1) * 4 + quad] = static_cast<uint8_t>(Eds1 + 127);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[Lay::bDsFull + pb]);
        cur = nxt;
      }
      if (!ok) break;
    }
    if (!ok) *abort_flag = 1;
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ / epilogue warps
    setmaxnreg_dec<Lay::kRegsDrain>();
    work.sleep = role_sleeps(kSleepMask, kRoleDrain);
    const int quad = warp & 3;
    const int row = quad * 32 + lane;                 // TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
    int it = 0, items = 0;
    bool ok = true;
    for (;;) {
      int g;
      int4 rec;
      if (!work.next(g, rec) || *abort_flag) break;
      const BwdItem w = decode_bwd(a, g, rec);
      BwdCursor cur;
      cur.begin(w);
      for (int n = 0; n < w.n_it; ++n, ++it, cur.advance(w)) {
        // dQ partial of (query head h, query tile qt) against this key tile,
        // this warp's 32 query rows: staged in shared memory and added to the
        // fp32 accumulator with TMA bulk reduce-adds.  Rows outside the
        // document carry exact zeros (their dS row is zero).
        if (!mbar_wait(&bars[Lay::bDqFull], it & 1, a.status, role_sleeps(kSleepMask, kRoleDrain))) { ok = false; break; }
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32x2_sync(tbase + lane_base + Lay::kTdQ, r0, tbase + lane_base + Lay::kTdQ + 32, r1);
        tc_fence_before();
        mbar_arrive(&bars[Lay::bDqEmpty]);
        if constexpr (kDet) {
          // Deterministic option: each partial becomes a 64-bit fixed-point
          // integer, and every lane adds its own query row with integer bulk
          // reduce-adds (32 columns per pass, one padded staging row), so the
          // sum does not depend on the order in which key tiles arrive.  Rows
          // outside the document are skipped (their partials are zero).
          const int qrow = cur.qt * kTile + 32 * quad + lane;
          unsigned long long* grow =
              reinterpret_cast<unsigned long long*>(a.dqacc) + ((w.s_doc + qrow) * a.Hq + cur.h) * D;
          uint8_t* slot = smem + Lay::kDQs + quad * Lay::kDqWarpBytes + lane * Lay::kDetRowBytes;
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const uint32_t (&r)[32] = p == 0 ? r0 : r1;
            bulk_wait_group_read<0>();           // this lane's previous reduce has read its row
#pragma unroll
            for (int k = 0; k < 16; ++k)
              *reinterpret_cast<ulonglong2*>(slot + 16 * k) =
                  make_ulonglong2(dq_fixed(__uint_as_float(r[2 * k])), dq_fixed(__uint_as_float(r[2 * k + 1])));
            fence_proxy_async_smem();
            if (qrow < w.L) bulk_reduce_add_u64(grow + 32 * p, slot, 256);
            bulk_commit_group();
          }
        } else {
          uint8_t* box0 = smem + Lay::kDQs + quad * Lay::kDqWarpBytes;
          uint8_t* box1 = box0 + Lay::kDqBoxBytes;
          // the reduce issued from these boxes one iteration ago has read them
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = lane * 128 + ((k ^ (lane & 7)) << 4);
            *reinterpret_cast<uint4*>(box0 + off) = make_uint4(r0[4 * k], r0[4 * k + 1], r0[4 * k + 2], r0[4 * k + 3]);
            *reinterpret_cast<uint4*>(box1 + off) = make_uint4(r1[4 * k], r1[4 * k + 1], r1[4 * k + 2], r1[4 * k + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int32_t y = static_cast<int32_t>(w.s_doc + cur.qt * kTile + 32 * quad);
            tma_reduce_add_2d(&a.tm_dq, cur.h * D, y, box0);
            tma_reduce_add_2d(&a.tm_dq, cur.h * D + 32, y, box1);
            bulk_commit_group();
          }
        }
      }
      if (!ok) break;
      // item epilogue: dV and dK rows (TMEM lane = key row), 1/sqrt(d) on dK
      if (!mbar_wait(&bars[Lay::bAccFull], items & 1, a.status, role_sleeps(kSleepMask, kRoleDrain))) { ok = false; break; }
      tc_fence_after();
      const int kj = w.kt * kTile + row;
      const int64_t orow = ((w.s_doc + kj) * a.Hkv + w.hk) * D;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        uint32_t r0[32], r1[32];
        tmem_ld32x2_sync(tbase + lane_base + (m ? Lay::kTdK : Lay::kTdV), r0,
                         tbase + lane_base + (m ? Lay::kTdK : Lay::kTdV) + 32, r1);
        if (m == 1) {
          tc_fence_before();
          mbar_arrive(&bars[Lay::bAccEmpty]);
        }
        if (kj < w.L) {
          __nv_bfloat16* dst = (m ? a.dk : a.dv) + orow;
          const float sc = m ? Lay::kInvSqrtD : 1.f;
          store_row_bf16_bits(dst, r0, sc);
          store_row_bf16_bits(dst + 32, r1, sc);
        }
      }
      ++items;
    }
    if (!ok) *abort_flag = 1;
    // every reduce-add has landed before the CTA exits (the deterministic
    // option's are issued by every lane)
    if (kDet || lane == 0) bulk_wait_group<0>();
  } else {
    setmaxnreg_dec<Lay::kRegsService>();
  }
  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    int it = 0, items = 0;
    ItemFeed feed{ring, a.plan_items, a.item_counter, total, a.Hkv, a.schedule == 0,
                  SnakeIter{0, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total}, 0, 0, a.status, role_sleeps(kSleepMask, kRoleProducer)};
    int4 rec;
    int g = feed.next(rec);
    bool ok = feed.publish(g, rec);
    while (ok && g >= 0 && !*abort_flag) {
      const BwdItem w = decode_bwd(a, g, rec);
      const int kb = items & 1;
      if (items >= 2 && !mbar_wait(&bars[Lay::bKVEmpty + kb], ((items >> 1) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleProducer))) { ok = false; break; }
      {
        // dQ = dS K: K's scale per 32-key group along the contraction (the
        // exact options fold K's exponents into dQ's payload: scale 1)
        uint32_t word = 0;
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const int rel = w.kt * kTile + gg * kBlock;
          const uint32_t byte = (!kExact && rel < w.L) ? __ldg(a.k_scales + static_cast<int64_t>(w.hk) * T + w.s_doc + rel) : 127u;
          word |= byte << (8 * gg);
        }
        reinterpret_cast<uint4*>(smem + Lay::kSfbDQ + kb * 512)[lane] = make_uint4(word, word, word, word);
      }
      if constexpr (kF4) {
        // the 4-bit S MMA's K scale words of this K/V buffer: row r, word i =
        // the four UE4M3 bytes of key row 32 i + r of the tile
        const int64_t k0 = w.s_doc + w.kt * kTile;
        uint32_t wk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t tt = k0 + 32 * i + lane;
          wk[i] = tt < T ? __ldg(reinterpret_cast<const uint32_t*>(a.k4_scales + (tt * a.Hkv + w.hk) * (D / 16))) : 0u;
        }
        reinterpret_cast<uint4*>(smem + Lay::kSk4 + kb * 512)[lane] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[Lay::bKVFull + kb], 2 * Lay::kTileBytes + (kF4 ? Lay::kTile4Bytes : 0));
        const int32_t y = static_cast<int32_t>(w.s_doc + w.kt * kTile);
        tma_load_2d(smem + Lay::kK + kb * Lay::kTileBytes, &a.tm_k, w.hk * D, y, &bars[Lay::bKVFull + kb]);
        tma_load_2d(smem + Lay::kV + kb * Lay::kTileBytes, &a.tm_v, w.hk * D, y, &bars[Lay::bKVFull + kb]);
        if constexpr (kF4)
          tma_load_2d(smem + Lay::kK4 + kb * Lay::kTile4Bytes, &a.tm_k4, w.hk * (D / 2), y, &bars[Lay::bKVFull + kb]);
      }
      __syncwarp();
      ++items;                         // K/V of this item are in flight
      // dV = P'^T dO and dK = dS^T Q contract over queries: the dO and Q
      // scale of each 32-query group, read one iteration ahead (lane gg < 4
      // reads group gg; the words are assembled with shuffles when used)
      auto load_scales = [&](const BwdCursor& c, uint32_t& bdo, uint32_t& bq) {
        const int rel = c.qt * kTile + (lane & 3) * kBlock;
        const int64_t idx = static_cast<int64_t>(c.h) * T + w.s_doc + min(rel, w.L - 1);
        bdo = __ldg(a.do_scales + idx);
        bq = __ldg(a.q_scales + idx);
        if (rel >= w.L) bdo = bq = 127u;
      };
      BwdCursor cur, nxt;
      cur.begin(w);
      nxt = cur;
      uint32_t bdo_next, bq_next;
      load_scales(cur, bdo_next, bq_next);
      for (int n = 0; n < w.n_it; ++n) {
        const int h = cur.h, qt = cur.qt;
        const uint32_t bdo = bdo_next, bq = bq_next;
        if (n + 1 < w.n_it) {
          nxt.advance(w);
          load_scales(nxt, bdo_next, bq_next);
        }
        const int st = it % Lay::kStages;
        if (it >= Lay::kStages &&
            !mbar_wait(&bars[Lay::bQDEmpty + st], ((it / Lay::kStages) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleProducer))) {
          ok = false;
          break;
        }
        uint32_t wdo = 0, wq = 0;
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          wdo |= __shfl_sync(0xffffffffu, bdo, gg) << (8 * gg);
          wq |= __shfl_sync(0xffffffffu, bq, gg) << (8 * gg);
        }
        // exact options: dO's and Q's exponents are folded into P' and dK's payload
        if constexpr (kExact) wdo = wq = 0x7f7f7f7fu;
        reinterpret_cast<uint4*>(smem + Lay::kSfbDV + st * 512)[lane] = make_uint4(wdo, wdo, wdo, wdo);
        reinterpret_cast<uint4*>(smem + Lay::kSfbDK + st * 512)[lane] = make_uint4(wq, wq, wq, wq);
        if constexpr (kF4) {
          // the 4-bit S MMA's Q scale words of this stage
          const int64_t q0 = w.s_doc + qt * kTile;
          uint32_t wq4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t tt = q0 + 32 * i + lane;
            wq4[i] = tt < T ? __ldg(reinterpret_cast<const uint32_t*>(a.q4_scales + (tt * a.Hq + h) * (D / 16))) : 0u;
          }
          reinterpret_cast<uint4*>(smem + Lay::kSq4 + st * 512)[lane] = make_uint4(wq4[0], wq4[1], wq4[2], wq4[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[Lay::bQDFull + st], 2 * Lay::kTileBytes + (kF4 ? Lay::kTile4Bytes : 0));
          const int32_t y = static_cast<int32_t>(w.s_doc + qt * kTile);
          tma_load_2d(smem + Lay::kQ + st * Lay::kTileBytes, &a.tm_q, h * D, y, &bars[Lay::bQDFull + st]);
          tma_load_2d(smem + Lay::kDO + st * Lay::kTileBytes, &a.tm_do, h * D, y, &bars[Lay::bQDFull + st]);
          if constexpr (kF4)
            tma_load_2d(smem + Lay::kQ4 + st * Lay::kTile4Bytes, &a.tm_q4, h * (D / 2), y, &bars[Lay::bQDFull + st]);
        }
        __syncwarp();
        ++it;
        cur = nxt;
      }
      if (!ok) break;
      // the next item is claimed once this one's last Q/dO loads are issued
      g = feed.next(rec);
      ok = feed.publish(g, rec);
    }
    if (!ok) *abort_flag = 1;
    // Let every copy still in flight land before the CTA can exit, also when
    // the loop ended because another warp gave up: the last phase armed on
    // each Q/dO stage and K/V buffer (already complete after a normal run).
    for (int x = (it > Lay::kStages ? it - Lay::kStages : 0); x < it; ++x)
      mbar_wait(&bars[Lay::bQDFull + (x % Lay::kStages)], (x / Lay::kStages) & 1, nullptr);
    for (int x = (items > 2 ? items - 2 : 0); x < items; ++x)
      mbar_wait(&bars[Lay::bKVFull + (x & 1)], (x >> 1) & 1, nullptr);
  } else if (warp >= 13) {
    // ------------------------------------------------------------ MMA issuers
    // Three issuing threads keep the tensor pipe fed: warp 13 issues S/dP,
    // warp 15 dQ, warp 14 the dV/dK accumulations, so no chain waits behind
    // another's blocked issue.  Each thread's commits track only its own
    // MMAs, so a barrier fed by two of them (ds_empty, kv_empty) counts one
    // arrival from each.
    if (lane == 0) {
      work.whole_warp = false;
      work.sleep = role_sleeps(kSleepMask, kRoleIssuer);
      // Shared-memory descriptors, computed once: a buffer's descriptor is its
      // base descriptor plus (byte offset >> 4) in the start-address field
      // (no carry out of the field: every address is below 228 KB).
      // Code tiles (64B swizzle, 512-byte row groups) serve both K-major
      // (S, dP: +32 bytes per K step) and MN-major (dQ, dV, dK: +32 rows =
      // 2048 bytes per K step) reads; P'/dS tiles use the 128B swizzle.
      const uint64_t dK0 = make_smem_desc(smem_u32(smem + Lay::kK), 16, 8 * D, Lay::kSwz);
      const uint64_t dV0 = make_smem_desc(smem_u32(smem + Lay::kV), 16, 8 * D, Lay::kSwz);
      const uint64_t dQ0 = make_smem_desc(smem_u32(smem + Lay::kQ), 16, 8 * D, Lay::kSwz);
      const uint64_t dDO0 = make_smem_desc(smem_u32(smem + Lay::kDO), 16, 8 * D, Lay::kSwz);
      const uint64_t dPp0 = make_smem_desc(smem_u32(smem + Lay::kPp), 16, 1024, kSwizzle128B);
      const uint64_t dDS0 = make_smem_desc(smem_u32(smem + Lay::kDS), 16, 1024, kSwizzle128B);
      // exact options: dQ reads its own payload tile
      const uint64_t dDQ0 = kExact ? make_smem_desc(smem_u32(smem + Lay::kDS2), 16, 1024, kSwizzle128B) : dDS0;
      const uint64_t dSF0 = make_smem_desc(smem_u32(smem + Lay::kSfaDV), 0, 128, kSwizzleNone);
      constexpr uint64_t kTileStep = Lay::kTileBytes >> 4, kPStep = Lay::kPTileBytes >> 4;
      constexpr uint64_t kKStep = 32 >> 4;                 // K-major: 32 bytes per K step
      constexpr uint64_t kMnStep = (32 * D) >> 4;          // MN-major code tile: 32 rows per K step
      constexpr uint64_t kMnStepP = (32 * kTile) >> 4;     // MN-major P'/dS tile: 32 rows per K step
      auto sf_desc = [&](int off) { return dSF0 + static_cast<uint64_t>((off - Lay::kSfaDV) >> 4); };
      int it = 0, items = 0;
      bool ok = true;
      int g;
      int4 rec;
      if (warp == 13) {
        // ---------------------------------------------- S and dP
        const uint32_t idesc_s = idesc_f8(128, 128, false, false);
        // S = Q K^T and dP = dO V^T from Q/dO stage st and K/V buffer kb
        auto issue_sdp = [&](int st, int kb) {
          const uint64_t q = dQ0 + st * kTileStep, dox = dDO0 + st * kTileStep;
          const uint64_t k = dK0 + kb * kTileStep, v = dV0 + kb * kTileStep;
          if constexpr (kF4) {
            // NVFP4 path: S recomputed with the forward's 4-bit MMA (same
            // operands, scales and K order; K = 64 in one instruction), dP
            // unscaled E4M3.  This stage's Q scale columns were last read by
            // S(it - 3) and the buffer's K scale columns by the item before
            // the previous one: both complete, since S(it - 1) completed
            // before the score warps released S/dP.
            tmem_cp_32x128b_x4(tbase + Lay::kTSq4 + 4 * st, sf_desc(Lay::kSq4 + st * 512));
            tmem_cp_32x128b_x4(tbase + Lay::kTSk4 + 4 * kb, sf_desc(Lay::kSk4 + kb * 512));
            const uint64_t q4 = make_smem_desc(smem_u32(smem + Lay::kQ4 + st * Lay::kTile4Bytes), 16, 8 * (D / 2), kSwizzle32B);
            const uint64_t k4 = make_smem_desc(smem_u32(smem + Lay::kK4 + kb * Lay::kTile4Bytes), 16, 8 * (D / 2), kSwizzle32B);
            mma_mxf4nvf4(tbase + Lay::kTS, q4, k4, idesc_mxf4nvf4(128, 128), tbase + Lay::kTSq4 + 4 * st,
                         tbase + Lay::kTSk4 + 4 * kb, 0u);
            mma_f8(tbase + Lay::kTdP, dox, v, idesc_s, 0u);
            mma_f8(tbase + Lay::kTdP, dox + kKStep, v + kKStep, idesc_s, 1u);
          } else {
            mma_f8_two_chains(tbase + Lay::kTS, q, q + kKStep, k, k + kKStep, tbase + Lay::kTdP, dox, dox + kKStep, v,
                              v + kKStep, idesc_s);
          }
          mma_commit(&bars[Lay::bSdpFull]);
        };
        bool have = work.next(g, rec) && !*abort_flag;
        BwdItem cur{};
        if (have) {
          cur = decode_bwd(a, g, rec);
          // first S/dP of the first item
          if (!mbar_wait(&bars[Lay::bKVFull + 0], 0, a.status, role_sleeps(kSleepMask, kRoleIssuer)) ||
              !mbar_wait(&bars[Lay::bQDFull + 0], 0, a.status, role_sleeps(kSleepMask, kRoleIssuer))) {
            ok = false;
            have = false;
          } else {
            tc_fence_after();
            issue_sdp(0, 0);
          }
        }
        while (have) {
          const int kb = items & 1;
          bool have_next = false;
          BwdItem nxt{};
          for (int n = 0; n < cur.n_it; ++n, ++it) {
            // 1. next S/dP (this item's next iteration, or the next item's
            //    first) once the compute warps have read S/dP(it)
            {
              int kb1 = kb;
              bool issue = false;
              if (n + 1 < cur.n_it) {
                issue = true;
              } else {
                have_next = work.next(g, rec) && !*abort_flag;
                if (have_next) {
                  nxt = decode_bwd(a, g, rec);
                  kb1 = (items + 1) & 1;
                  if (!mbar_wait(&bars[Lay::bKVFull + kb1], ((items + 1) >> 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
                  issue = true;
                }
              }
              if (issue) {
                const int st1 = (it + 1) % Lay::kStages;
                if (!mbar_wait(&bars[Lay::bQDFull + st1], ((it + 1) / Lay::kStages) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
                if (!mbar_wait(&bars[Lay::bSdpEmpty], it & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
                tc_fence_after();
                issue_sdp(st1, kb1);
              }
            }
          }
          if (!ok) break;
          // S and dP were this buffer's readers on this thread (dQ commits its own arrival)
          mma_commit(&bars[Lay::bKVEmpty + kb]);
          ++items;
          if (!have_next) break;
          cur = nxt;
        }
      } else if (warp == 15) {
        // ---------------------------------------------- dQ
        constexpr uint32_t iq0 = idesc_mxf8(128, D, false, true, 0, 0), iq1 = idesc_mxf8(128, D, false, true, 1, 1);
        constexpr uint32_t iq2 = idesc_mxf8(128, D, false, true, 2, 2), iq3 = idesc_mxf8(128, D, false, true, 3, 3);
        for (;;) {
          if (!work.next(g, rec) || *abort_flag) break;
          const BwdItem w = decode_bwd(a, g, rec);
          const int kb = items & 1;
          const uint64_t kdesc = dK0 + kb * kTileStep;
          const uint32_t tsfb_dq = tbase + Lay::kTSfbDQ + 4 * kb;
          for (int n = 0; n < w.n_it; ++n, ++it) {
            const int pb = it & 1;
            const uint32_t tset = tbase + Lay::kTSet + Lay::kSetCols * pb;
            const uint64_t dsd = dDQ0 + pb * kPStep;
            // dQ(it) = dS K   (A: dS K-major, B: K MN-major), once dS(it) and
            // its scale words are in shared memory (S/dP(it) completed, so
            // K/V of this item have landed) and dQ(it-1) has been read.
            // Passing ds_full(it) also means the MMAs of it-2, the last
            // readers of this parity's scale columns, are complete: the
            // compute warps waited for them before writing dS(it).
            if (!mbar_wait(&bars[Lay::bDsFull + pb], (it >> 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
            if (it > 0 && !mbar_wait(&bars[Lay::bDqEmpty], (it - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
            tc_fence_after();
            if (n == 0) tmem_cp_32x128b_x4(tsfb_dq, sf_desc(Lay::kSfbDQ + kb * 512));
            tmem_cp_32x128b_x4(tset + Lay::kSfaDQo, sf_desc(Lay::kSfaDQ + pb * 512));
            mma_mxf8_chain4(tbase + Lay::kTdQ, dsd, dsd + kKStep, dsd + 2 * kKStep, dsd + 3 * kKStep, kdesc,
                            kdesc + kMnStep, kdesc + 2 * kMnStep, kdesc + 3 * kMnStep, iq0, iq1, iq2, iq3,
                            tset + Lay::kSfaDQo, tsfb_dq, 0u);
            mma_commit(&bars[Lay::bDqFull]);
            mma_commit(&bars[Lay::bDsEmpty + pb]);
          }
          if (!ok) break;
          mma_commit(&bars[Lay::bKVEmpty + kb]);        // K was read by dQ
          ++items;
        }
      } else {
        // ---------------------------------------------- dV and dK
        // P' operand of dV: constant scale 2^-8, copied to tensor memory once
        // (the exact options' scale words are written per iteration by the
        // score warps in the same place)
        if constexpr (!kExact) {
          const uint32_t pword = 0x77777777u;  // 119 = 127 - 8 in every byte
          uint32_t* sfa_dv = reinterpret_cast<uint32_t*>(smem + Lay::kSfaDV);
          for (int i = 0; i < 128; ++i) sfa_dv[i] = pword;
          fence_proxy_async_smem();
          tmem_cp_32x128b_x4(tbase + Lay::kTSfaDV, sf_desc(Lay::kSfaDV));
        }
        constexpr uint32_t iv0 = idesc_mxf8(128, D, true, true, 0, 0), iv1 = idesc_mxf8(128, D, true, true, 1, 1);
        constexpr uint32_t iv2 = idesc_mxf8(128, D, true, true, 2, 2), iv3 = idesc_mxf8(128, D, true, true, 3, 3);
        for (;;) {
          if (!work.next(g, rec) || *abort_flag) break;
          const BwdItem w = decode_bwd(a, g, rec);
          for (int n = 0; n < w.n_it; ++n, ++it) {
            const int st = it % Lay::kStages;
            const int pb = it & 1;
            const uint32_t tset = tbase + Lay::kTSet + Lay::kSetCols * pb;
            const uint64_t ppd = dPp0 + pb * kPStep, dsd = dDS0 + pb * kPStep;
            const uint64_t qd = dQ0 + st * kTileStep, dod = dDO0 + st * kTileStep;
            // P'(it), dS(it) and their scale words are in shared memory (and
            // S/dP(it) completed, so Q/dO of this stage have landed); from an
            // item's first iteration on, the previous item's epilogue must
            // have read dV/dK
            if (!mbar_wait(&bars[Lay::bDsFull + pb], (it >> 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
            if (n == 0 && items > 0 && !mbar_wait(&bars[Lay::bAccEmpty], (items - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) {
              ok = false;
              break;
            }
            tc_fence_after();
            tmem_cp_32x128b_x4(tset + Lay::kSfbDVo, sf_desc(Lay::kSfbDV + st * 512));
            // exact options: P''s scale per 32-query block, this parity's words
            if constexpr (kExact) tmem_cp_32x128b_x4(tset + Lay::kSfaDVo, sf_desc(Lay::kSfaDV + pb * 512));
            tmem_cp_32x128b_x4(tset + Lay::kSfaDKo, sf_desc(Lay::kSfaDK + pb * 512));
            tmem_cp_32x128b_x4(tset + Lay::kSfbDKo, sf_desc(Lay::kSfbDK + st * 512));
            const uint32_t acc_on = (n > 0) ? 1u : 0u;
            // dV += P'^T dO   (A: P' viewed MN-major, B: dO MN-major)
            mma_mxf8_chain4(tbase + Lay::kTdV, ppd, ppd + kMnStepP, ppd + 2 * kMnStepP, ppd + 3 * kMnStepP, dod,
                            dod + kMnStep, dod + 2 * kMnStep, dod + 3 * kMnStep, iv0, iv1, iv2, iv3,
                            kExact ? tset + Lay::kSfaDVo : tbase + Lay::kTSfaDV, tset + Lay::kSfbDVo, acc_on);
            // dK += dS^T Q
            mma_mxf8_chain4(tbase + Lay::kTdK, dsd, dsd + kMnStepP, dsd + 2 * kMnStepP, dsd + 3 * kMnStepP, qd,
                            qd + kMnStep, qd + 2 * kMnStep, qd + 3 * kMnStep, iv0, iv1, iv2, iv3,
                            tset + Lay::kSfaDKo, tset + Lay::kSfbDKo, acc_on);
            mma_commit(&bars[Lay::bDsEmpty + pb]);
            // the last readers of this Q/dO stage (S/dP(it) completed before ds_full(it))
            mma_commit(&bars[Lay::bQDEmpty + st]);
          }
          if (!ok) break;
          mma_commit(&bars[Lay::bAccFull]);
          ++items;
        }
      }
      if (!ok) *abort_flag = 1;
      // every MMA this thread issued completes before TMEM is freed
      uint64_t* fin = &bars[warp == 13 ? Lay::bFinal : (warp == 14 ? Lay::bFinal2 : Lay::bFinal3)];
      mma_commit(fin);
      mbar_wait(fin, 0, nullptr);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 13) tmem_dealloc(tbase, 512);
}

template <bool kDump, bool kDet = false, bool kExact = false, bool kF4 = false>
static void launch_bwd64_t(const BwdArgs& a, int num_ctas, cudaStream_t st) {
  constexpr int smem = Bwd64LayoutT<kExact, kF4>::kSmemAlloc;
  static std::atomic<uint64_t> configured{0};
  if (first_use_on_device(configured))
    cudaFuncSetAttribute(bwd64_kernel<kDump, kDet, kExact, kF4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  bwd64_kernel<kDump, kDet, kExact, kF4><<<num_ctas, Bwd64Layout::kThreads, smem, st>>>(a);
}

cudaError_t launch_bwd_d64(const BwdArgs& a, int num_ctas, cudaStream_t st) {
  // the dump variant (a diagnostic) when a score-tile copy is requested (the
  // host rejects it together with the deterministic, exact or NVFP4 options)
  if (a.dump.s != nullptr) {
    launch_bwd64_t<true>(a, num_ctas, st);
  } else if (a.exact) {
    if (a.det_dq) launch_bwd64_t<false, true, true>(a, num_ctas, st);
    else launch_bwd64_t<false, false, true>(a, num_ctas, st);
  } else if (a.nvfp4) {
    if (a.det_dq) launch_bwd64_t<false, true, false, true>(a, num_ctas, st);
    else launch_bwd64_t<false, false, false, true>(a, num_ctas, st);
  } else if (a.det_dq) {
    launch_bwd64_t<false, true>(a, num_ctas, st);
  } else {
    launch_bwd64_t<false>(a, num_ctas, st);
  }
  return cudaGetLastError();
}

}  // namespace flamia
