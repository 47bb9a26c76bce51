// MXFP8 causal packed attention forward for sm_103a.
//
// Method: FLAMIA (arXiv 2611.03344) Sections 3.4-3.6 and Appendix B.1.
//   S = Qhat Khat^T on E4M3 codes with an unscaled tcgen05 MMA; the token-block
//   scales factor out of the dot product (Section 3.5.1), so the row factor
//   2^{E_Q(i)} log2(e)/sqrt(d) and the per-32-key column factor 2^{E_K(g)} are
//   folded into one multiply per score in the softmax warps.
//   Online softmax in fp32, per query row, with conditional rescaling: the
//   running maximum m only moves when a tile raises it by more than tau (log2
//   units); P-hat = E4M3(2^{S2 - m + c}) is written to shared memory and
//   O += P-hat Vhat runs as a UE8M0 block-scaled MMA (P-hat scale 2^-c, V
//   scale per 32-key token block), accumulating in tensor memory.
//   Key tiles of 128 document-relative keys are visited from the highest
//   fully visible tile down to tile 0, and the diagonal tile of a causal
//   call last.
//
// Exact options (fwd_kernel<d, true>; Section 3.2 and Appendix A.3): Q, K, V
// carry one exponent per token.
//   * S is a UE8M0 block-scaled MMA with K's per-key scales; Q's exponent
//     stays in the row factor.
//   * V's per-key exponent is folded into P-hat on the diagonal tile of a
//     causal call (the pages' choice): for that tile's K/V stage the
//     producer writes a table of fold factors 2^(b_j - s_g - c), the P-hat
//     scale byte s_g of each 32-key group, and the prefix maxima of the V
//     bytes.  The softmax multiplies each probability by its key's factor
//     and writes its row's four P-hat scale bytes (the group holding the
//     row takes its scale from the prefix maximum up to the row); the PV
//     issuer copies those bytes into TMEM before the MMA.
//   * The tiles before it hold only keys every row of the tile sees: they
//     multiply a token-block copy of V with the fixed 2^c, as the default
//     path does.
// No scale then depends on a key the row does not see.
//
// Work: one item = (query head, document, 128-query tile).  A persistent grid
// walks the device-built longest-first list in snake order.
//
// Warp roles (256 threads; d = 64: two CTAs per SM with 256 TMEM columns and
// one S buffer each, d = 128: one CTA per SM with 512 columns):
//   warps 0-3  softmax: thread i owns query row i (TMEM lane i)
//   warp 4     TMA producer: Q tile per item, K/V tiles through a 3-stage ring,
//              and the V block-scale words for the MMA
//   warp 5     S issuer (lane 0) and TMEM owner
//   warp 6     PV issuer (lane 0)
//   warp 7     (d = 64) clears the backward's fp32 dQ accumulator rows of
//              every item with TMA stores of a zero box: the forward leaves
//              the memory system mostly idle, so the clearing is nearly free
// TMEM columns: S (one or two 128-column buffers), then O (d columns), the
//   P-hat scales (4 columns) and the V scales (4 columns per ring stage).
//
// Pipeline invariants (every mbarrier is waited on in the order its phases
// complete, so parity waits never alias):
//   q_full/q_empty      one phase per item
//   kv_full/kv_empty    one phase per use of a ring stage
//   s_full/s_empty      one phase per use of an S buffer
//   p_full/pv_done      one phase per use of a P-hat buffer (tile t uses
//                       buffer t & 1); the softmax waits pv_done for tile t-2
//                       before rewriting a buffer, for tile t-1 only when it
//                       must rescale O, and for its last tile in the epilogue
//   o_empty             one phase per item (epilogue has read O)
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "flamia_common.cuh"
#include "launch.h"

namespace flamia {

template <int D, bool kExact = false, bool kF4 = false>
struct FwdLayout {
  static constexpr int kStages = 3;
  static constexpr int kTileBytes = kTile * D;
  static constexpr uint32_t kSwz = (D == 64) ? kSwizzle64B : kSwizzle128B;
  static constexpr int kQ = 0;                                 // two Q buffers (items alternate)
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;        // two P-hat buffers
  static constexpr int kSfa = kP + 2 * kTile * kTile;
  static constexpr int kSfb = kSfa + 512;
  // 4 KB of zeros (d = 64): the source of the TMA stores that clear the
  // backward's fp32 dQ accumulator, one 32 x 32 box at a time
  static constexpr int kZero = (kSfb + kStages * 512 + 1023) / 1024 * 1024;
  static constexpr int kZeroBytes = (D == 64) ? 4096 : 0;
  // exact options: the S MMA's scale words (Q: constant 1; K: the per-key
  // scale of each key of a stage), the V fold table of each stage (per key:
  // fp32 fold factor, V scale byte, prefix maximum of the V bytes within its
  // 32-key group; the P-hat scale word of fully visible groups) and the P-hat
  // scale words of each P-hat buffer, one per query row
  static constexpr int kSqa = kZero + kZeroBytes;
  static constexpr int kSkb = kSqa + 512;
  static constexpr int kVt = kSkb + kStages * 512;
  static constexpr int kVtBytes = 1024;
  static constexpr int kVtColf = 0, kVtBytesV = 512, kVtPm = 640, kVtPword = 768;
  static constexpr int kSpa = kVt + kStages * kVtBytes;
  // NVFP4 option: the 4-bit S MMA's scale words of Q (per Q buffer) and K
  // (per stage), one 512-byte block per 64-element chunk of the head
  // dimension (row r, word i = the four UE4M3 bytes of operand row 32 i + r),
  // and the log-domain P-hat scale words of each P-hat buffer
  static constexpr int kC4 = D / 64;
  static constexpr int kSq4 = kZero + kZeroBytes;
  static constexpr int kSk4 = kSq4 + 2 * kC4 * 512;
  static constexpr int kSpa4 = kSk4 + kStages * kC4 * 512;
  static constexpr int kPsw = kF4 ? kSpa4 : kSpa;                 // per-row P-hat scale words
  static constexpr int kBar = kExact ? kSpa + 2 * 512 : (kF4 ? kSpa4 + 2 * 512 : kZero + kZeroBytes);
  enum {
    bQFull = 0,                // per Q buffer
    bQEmpty = bQFull + 2,      // per Q buffer
    bKVFull = bQEmpty + 2,
    bKVEmpty = bKVFull + kStages,
    bSFull = bKVEmpty + kStages,
    bSEmpty = bSFull + 2,
    bPFull = bSEmpty + 2,      // per P-hat buffer: softmax wrote it
    bPVDone = bPFull + 2,      // per P-hat buffer: the PV MMA reading it has completed
    bOEmpty = bPVDone + 2,
    bFinal,
    bFinal2,
    kNumBars
  };
  static constexpr int kSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kSlot + 8;
  static constexpr int kRing = (kAbort + 16 + 15) / 16 * 16;   // work hand-out ring (ItemRing)
  static constexpr int kBytes = kRing + static_cast<int>(sizeof(ItemRing));
  static constexpr int kSmemAlloc = kBytes + 1024;
  // d = 64 runs two CTAs per SM, each with one S buffer in 256 TMEM columns
  // (S 128 + O 64 + scale factors), so every SM sub-partition holds two softmax
  // warps; d = 128 needs 512 columns (double-buffered S + O 128) and runs one.
  static constexpr int kCtasPerSm = (D == 64) ? 2 : 1;
  static constexpr int kSBufs = (D == 64) ? 1 : 2;
  static constexpr uint32_t kTmemCols = (D == 64) ? 256 : 512;
  // 256 threads: the softmax warpgroup and a service warpgroup (producer, S
  // issuer, PV issuer, one idle warp).  At d = 64 (two CTAs per SM, 128
  // registers per thread at launch) the service warpgroup gives registers to
  // the softmax warps with setmaxnreg: 2 x (200 + 56) x 128 = the SM's 65536.
  static constexpr int kThreads = 256;
  static constexpr uint32_t kRegsSoftmax = 200, kRegsService = 56;
  static_assert(D != 64 || (kRegsSoftmax + kRegsService) * 128 * kCtasPerSm <= 65536, "register split");
  static constexpr uint32_t kTS = 0;
  static constexpr uint32_t kTO = kSBufs * 128;
  static constexpr uint32_t kTSfa = kTO + D;
  // P-hat scale columns: the constant 2^-c words (4 columns), and with the
  // options the per-row words of each P-hat buffer (exact: 4 more columns
  // after the constant, which their off-diagonal tiles still use; NVFP4: in
  // place of it)
  static constexpr uint32_t kTSfb = kTSfa + (kExact ? 12 : 8);
  // exact options: S MMA scale factors (Q constant, K per stage)
  static constexpr uint32_t kTSqa = kTSfb + 4 * kStages;
  static constexpr uint32_t kTSkb = kTSqa + 4;
  static_assert(!kExact || kTSkb + 4 * kStages <= kTmemCols, "TMEM columns");
  // NVFP4 option: the 4-bit S MMA's scale factors (Q per Q buffer, K per stage)
  static constexpr uint32_t kTSq4 = kTSfb + 4 * kStages;
  static constexpr uint32_t kTSk4 = kTSq4 + 2 * 4 * kC4;
  static_assert(!kF4 || kTSk4 + 4 * kStages * kC4 <= kTmemCols, "TMEM columns");
  static_assert(!(kF4 && kExact), "the NVFP4 path and the exact options are separate");
  static_assert(kCtasPerSm * (kSmemAlloc + 1024) <= 233472, "shared memory per SM");
  // log2(e) / sqrt(d)
  static constexpr float kSmScale = (D == 64) ? 0.18033688011112042f : 0.12751743082459868f;
};

struct FwdItem {
  int h, hk, doc, qt, n_kt, nt;
  int64_t s_doc;
  int L;
};

// item g = u * Hq + h with plan record rec = {doc, cost c, first token, length}
__device__ __forceinline__ FwdItem decode_fwd(const FwdArgs& a, int g, int4 rec) {
  FwdItem it;
  it.h = g % a.Hq;
  it.hk = it.h / (a.Hq / a.Hkv);
  it.doc = rec.x;
  it.s_doc = rec.z;
  it.L = rec.w;
  it.nt = (it.L + kTile - 1) / kTile;
  it.qt = rec.y - 1;
  it.n_kt = a.causal ? it.qt + 1 : it.nt;
  return it;
}

// Key tile visited at step j: causal calls take the fully visible tiles
// qt-1 .. 0 and the diagonal tile qt last; non-causal calls nt-1 .. 0.
__device__ __forceinline__ int fwd_key_tile(const FwdItem& it, int j, int causal) {
  if (causal) return j == it.n_kt - 1 ? it.qt : it.qt - 1 - j;
  return it.nt - 1 - j;
}

template <int D, bool kExact, bool kDump = false, bool kF4 = false>
__global__ void __launch_bounds__(FwdLayout<D>::kThreads, FwdLayout<D>::kCtasPerSm) fwd_kernel(const __grid_constant__ FwdArgs a) {
  using Lay = FwdLayout<D, kExact, kF4>;
  // Roles that sleep in their waits.  Polling warps take issue slots from the
  // softmax warps on their sub-partition; sleeping ones wake a little later.
  // Measured: every role sleeping makes the default forward 2.6 % faster, the
  // exact options' forward (whose diagonal tile waits on the producer's fold
  // table) 3.5 % slower, where only the producer's sleeping is neutral.
  constexpr unsigned kSleepMask = kExact ? kRoleProducer : (kRoleProducer | kRoleIssuer | kRoleCompute | kRoleDrain);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Lay::kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[Lay::bQFull + b], 1);
      mbar_init(&bars[Lay::bQEmpty + b], 1);
    }
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&bars[Lay::bKVFull + s], 1);
      mbar_init(&bars[Lay::bKVEmpty + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[Lay::bSFull + b], 1);
      mbar_init(&bars[Lay::bSEmpty + b], 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[Lay::bPFull + b], 128);
      mbar_init(&bars[Lay::bPVDone + b], 1);
    }
    mbar_init(&bars[Lay::bOEmpty], 128);
    mbar_init(&bars[Lay::bFinal], 1);
    mbar_init(&bars[Lay::bFinal2], 1);
    // consumers of the item ring: the four softmax warps, the S and PV
    // issuers and warp 7
    reinterpret_cast<ItemRing*>(smem + Lay::kRing)->init(7);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tslot, Lay::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&a.tm_q);
    tma_prefetch_desc(&a.tm_k);
    tma_prefetch_desc(&a.tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  const int valid_plan = __ldg(a.plan_hdr + 2);
  const int total = valid_plan ? __ldg(a.plan_hdr + 0) * a.Hq : 0;
  ItemRing* ring = reinterpret_cast<ItemRing*>(smem + Lay::kRing);
  // every role reads its items from the ring the producer fills
  ItemReader work{ring, abort_flag, a.status, 0, true};
  const int64_t T = a.T;

  if (warp < 4) {
    // ------------------------------------------------------------ softmax
    if constexpr (D == 64) setmaxnreg_inc<Lay::kRegsSoftmax>();
    work.sleep = role_sleeps(kSleepMask, kRoleCompute);
    const int row = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    uint8_t* sP = smem + Lay::kP;
    const float tau = a.tau;
    // the NVFP4 path quantizes P-hat in the log domain: no fixed 2^c
    const float cexp = kF4 ? 0.f : static_cast<float>(a.c_exp);
    // rotated Q and K (Hadamard option): Q_r K_r^T = d Q K^T, and 1/d is exact
    const float sm_scale = a.hadamard ? Lay::kSmScale * (1.f / D) : Lay::kSmScale;
    int it = 0;
    // The epilogue of an item (O = acc * 2^c / l16, LSE = (m + log2 l16 - c)
    // ln 2) runs once the next item's first P-hat tile is written, so the wait
    // for the item's last PV overlaps that tile's work instead of stalling
    // the warp.  The next item's first PV waits for it (o_empty).
    struct Pending {
      int64_t t;
      float m, l16;
      int h, pv;
      bool on, valid;
    } pend{0, 0.f, 0.f, 0, 0, false, false};
    bool o_store_pending = false;     // an O store of this warp may still be reading its staging rows
    auto epilogue = [&](const Pending& e) -> bool {
      if (!mbar_wait(&bars[Lay::bPVDone + (e.pv & 1)], (e.pv >> 1) & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) return false;
      tc_fence_after();
      const float inv = ldexpf(1.f, kF4 ? 0 : a.c_exp) / e.l16;
      // d = 64 with the exact options or the NVFP4 path: a warp whose 32 rows
      // all lie in the document hands them to the TMA unit as one 32 x 64 box
      // (bf16, 128B swizzle), staged in its rows of the P-hat buffer of the
      // item's last tile: that tile's PV has completed, and the buffer's next
      // P-hat write waits for the store to have read it.  Plain stores take
      // the rows of a warp at the document end.  (Measured: the TMA stores
      // make those two forwards 3-4 % faster and the default one 4 % slower,
      // which keeps plain stores.)
      const bool tma_rows = D == 64 && (kExact || kF4) && __all_sync(0xffffffffu, e.valid);
      if (tma_rows) {
        uint8_t* scr = sP + (e.pv & 1) * (kTile * kTile) + warp * 32 * 128;
        uint32_t r0[32], r1[32];
        tmem_ld32x2_sync(tbase + lane_base + Lay::kTO, r0, tbase + lane_base + Lay::kTO + 32, r1);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t (&r)[32] = k < 4 ? r0 : r1;
          const int kk = (k & 3) * 8;
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(r[kk + 2 * q]) * inv,
                                                      __uint_as_float(r[kk + 2 * q + 1]) * inv);
            pk[q] = *reinterpret_cast<uint32_t*>(&p2);
          }
          *reinterpret_cast<uint4*>(scr + lane * 128 + ((k ^ (lane & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // lane 0 holds the warp's first row
          tma_store_2d(&a.tm_o, e.h * D, static_cast<int32_t>(e.t), scr);
          bulk_commit_group();
        }
        o_store_pending = true;
      } else {
        // O row, 32 columns at a time: scale, round to bf16, store
        uint4* dst = reinterpret_cast<uint4*>(a.out + (e.t * a.Hq + e.h) * D);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32_sync(tbase + lane_base + Lay::kTO + 32 * cc, r);
          if (e.valid) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t pk[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(r[8 * k + 2 * q]) * inv,
                                                          __uint_as_float(r[8 * k + 2 * q + 1]) * inv);
                pk[q] = *reinterpret_cast<uint32_t*>(&p2);
              }
              dst[4 * cc + k] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[Lay::bOEmpty]);
      if (e.valid) a.lse[static_cast<int64_t>(e.h) * T + e.t] = (e.m + log2f(e.l16) - cexp) * kLn2;
      return true;
    };
    for (;;) {
      int g;
      int4 rec;
      if (!work.next(g, rec) || *abort_flag) break;
      const FwdItem w = decode_fwd(a, g, rec);
      const int qi = w.qt * kTile + row;
      const bool valid = qi < w.L;
      const int64_t t = w.s_doc + qi;
      // Q's token-block exponent (the NVFP4 path's scales are inside the S MMA)
      const int eq = (!kF4 && valid) ? static_cast<int>(__ldg(a.q_scales + static_cast<int64_t>(w.h) * T + t)) - 127 : 0;
      float m = -INFINITY, l16 = 0.f;
      bool ok = true;
      // K block scales of the next key tile, loaded one tile ahead so their
      // latency hides behind the current tile's work
      const uint8_t* ksc = a.k_scales + static_cast<int64_t>(w.hk) * T + w.s_doc;
      // raw bytes, loaded from an index clamped into the document; a group
      // past the document end is given scale 1 only where it is used
      auto load_k_scales = [&](int kt, uint32_t (&e)[4]) {
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) e[gg] = __ldg(ksc + min(kt * kTile + gg * kBlock, w.L - 1));
      };
      uint32_t ek_next[4];
      if constexpr (!kExact && !kF4) load_k_scales(fwd_key_tile(w, 0, a.causal), ek_next);
      for (int j = 0; j < w.n_kt; ++j, ++it) {
        const int kt = fwd_key_tile(w, j, a.causal);
        float cg[4];
        if constexpr (kExact || kF4) {
          // the per-key K scales (exact options) or the NVFP4 scales of Q and
          // K are applied inside the S MMA
          const float c0 = scale_pow2(sm_scale, eq);
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) cg[gg] = c0;
        } else {
#pragma unroll
          for (int gg = 0; gg < 4; ++gg)
            cg[gg] = scale_pow2(sm_scale, eq + (kt * kTile + gg * kBlock < w.L ? static_cast<int>(ek_next[gg]) - 127 : 0));
          if (j + 1 < w.n_kt) load_k_scales(fwd_key_tile(w, j + 1, a.causal), ek_next);
        }
        // visible keys of this row.  A row past the document end is left
        // unmasked: its O row and LSE are never stored, and its P-hat row
        // only feeds that O row.
        int nvis;
        if (!valid) nvis = kTile;
        else if (a.causal) nvis = (kt == w.qt) ? row + 1 : kTile;
        else nvis = min(kTile, w.L - kt * kTile);

        const int b = it & 1;                                    // P-hat buffer
        const int sb = Lay::kSBufs == 2 ? (it & 1) : 0;          // S buffer
        const uint32_t sph = Lay::kSBufs == 2 ? ((it >> 1) & 1) : (it & 1);
        if (!mbar_wait(&bars[Lay::bSFull + sb], sph, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
        tc_fence_after();
        // Masked scores (beyond the causal diagonal or the document end)
        // become -inf in place: they never win the maximum and their
        // exponential is an exact 0, so partial tiles share the code of fully
        // visible ones.  On fully visible tiles the TMEM loads themselves
        // return each 32-key group's maximum (tcgen05.ld.red).
        const bool full = __all_sync(0xffffffffu, nvis == kTile);
        uint32_t sv[128];
        float gmx[4];
        {
          uint32_t (&c0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
          uint32_t (&c1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
          uint32_t (&c2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[64]);
          uint32_t (&c3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[96]);
          // one wait for the four loads; the group maxima of partial tiles
          // are recomputed below over the visible scores
          tmem_ld32x4_max_sync(tbase + lane_base + Lay::kTS + sb * 128, c0, c1, c2, c3, gmx);
        }
        tc_fence_before();
        mbar_arrive(&bars[Lay::bSEmpty + sb]);
        if constexpr (kDump) {
          // diagnostic copy of the raw S tile and the row's group factors
          if (w.h == a.dump.h && w.doc == a.dump.doc && w.qt == a.dump.qt && kt == a.dump.kt) {
#pragma unroll
            for (int c = 0; c < kTile; ++c) a.dump.s[row * kTile + c] = __uint_as_float(sv[c]);
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) a.dump.f[row * 4 + gg] = cg[gg];
          }
        }
        if (!full) {
#pragma unroll
          for (int c = 0; c < kTile; ++c)
            if (c >= nvis) sv[c] = 0xff800000u;
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            float gm = __uint_as_float(sv[32 * gg]);
#pragma unroll
            for (int c = 1; c < 31; c += 2)
              gm = max3f(gm, __uint_as_float(sv[32 * gg + c]), __uint_as_float(sv[32 * gg + c + 1]));
            gmx[gg] = fmaxf(gm, __uint_as_float(sv[32 * gg + 31]));
          }
        }
        // row maximum of the visible scores S2 = acc * c_g (log2 units), taken
        // on the raw accumulators per 32-key group (c_g > 0 and rounding are
        // monotone, so max(acc) * c_g equals max(acc * c_g))
        float tmax = -INFINITY;
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) tmax = fmaxf(tmax, gmx[gg] * cg[gg]);
        const bool upd = valid && (m == -INFINITY || tmax - m > tau);
        float alpha = 1.f;
        if (upd) {
          alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - tmax);
          m = tmax;
        }
        // O may only be rescaled once the previous tile's PV has completed.
        // tcgen05.ld/st are warp-collective: the whole warp rescales its 32
        // rows when any of them moved its maximum (alpha = 1 for the others).
        if (j > 0) {
          if (__any_sync(0xffffffffu, upd)) {
            const int pv = it - 1;
            if (!mbar_wait(&bars[Lay::bPVDone + (pv & 1)], (pv >> 1) & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < D / 16; ++cc) {
              uint32_t o[16];
              const uint32_t oaddr = tbase + lane_base + Lay::kTO + 16 * cc;
              tmem_ld16_sync(oaddr, o);
#pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st16(oaddr, o);
            }
            tmem_wait_st();
          }
          l16 *= alpha;
        }
        // the P-hat buffer of this tile was last read by the PV of tile it-2
        if (it >= 2 && !mbar_wait(&bars[Lay::bPVDone + b], ((it >> 1) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
        // and perhaps, in this warp's rows, by the TMA store of an item's O
        if (o_store_pending) {
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
          o_store_pending = false;
        }
        // probabilities, scaled by 2^c, rounded to E4M3, row r of P-hat in
        // the 128B-swizzled K-major layout the MMA reads
        // a row past the document end never sets m; offset 0 keeps its
        // (never stored) values finite or +inf, which the conversion saturates
        const float negm = m == -INFINITY ? 0.f : cexp - m;
        float lsum = 0.f;
        const uint32_t rbase = b * (kTile * kTile) + (row >> 3) * 1024 + (row & 7) * 128;
        // exact options: V's per-key exponent folded into P-hat.  The stage's
        // table holds, per key j, f_j = 2^(b_j - s_g - c) for the P-hat scale
        // byte s_g = max(G_g - c, 0) of its 32-key group (G_g the largest V
        // byte of the group's keys in the document); on the diagonal tile the
        // group holding this row's own position takes its scale from the
        // prefix maximum up to the row instead (keys past the row are masked).
        const uint8_t* vt = smem + Lay::kVt + (it % Lay::kStages) * Lay::kVtBytes;
        int dgrp = -1, sdiag = 0;
        uint32_t pword = 0;
        // exact options: the fold runs on the diagonal tile of a causal call
        // only; the tiles before it multiply V's token-block codes like the
        // default path (P-hat scale 2^-c)
        const bool vfold = kExact && a.causal && kt == w.qt;
        if constexpr (kExact) if (vfold) {
          const int st = it % Lay::kStages;
          // acquire the producer's table writes for this stage (long complete)
          if (!mbar_wait(&bars[Lay::bKVFull + st], (it / Lay::kStages) & 1, a.status, role_sleeps(kSleepMask, kRoleCompute))) { ok = false; break; }
          pword = *reinterpret_cast<const uint32_t*>(vt + Lay::kVtPword);
          {
            dgrp = row >> 5;                     // uniform across the warp
            sdiag = max(static_cast<int>(vt[Lay::kVtPm + row]) - a.c_exp, 0);
            pword = (pword & ~(0xffu << (8 * dgrp))) | (static_cast<uint32_t>(sdiag) << (8 * dgrp));
          }
          reinterpret_cast<uint32_t*>(smem + Lay::kSpa + b * 512)[(row & 31) * 4 + (row >> 5)] = pword;
        }
        // NVFP4 path: log-domain P-hat (Section 3.5.2).  Each 32-key group
        // takes E_g, the round-up exponent of its largest probability
        // 2^(max S2 - m); its codes are E4M3(2^(S2 - m - E_g)) with block
        // scale 2^E_g (no saturation), and the row sum adds each group's
        // unquantized probabilities back at 2^E_g.
        float goff[4], gsc[4];
        if constexpr (kF4) {
          uint32_t pw4 = 0;
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            const float pmax = ex2_approx(fmaf(gmx[gg], cg[gg], negm));
            const int E = roundup_exponent_from_bits(__float_as_uint(pmax));
            goff[gg] = negm - static_cast<float>(E);
            gsc[gg] = pow2f(E);
            pw4 |= static_cast<uint32_t>(E + 127) << (8 * gg);
          }
          reinterpret_cast<uint32_t*>(smem + Lay::kSpa4 + b * 512)[(row & 31) * 4 + (row >> 5)] = pw4;
        }
        {
          // the probability loop, in two copies for the exact options: with
          // the V fold (their diagonal tile) and without it (every other tile)
          auto prob_loop = [&](auto fold_tag) {
            constexpr bool kFold = decltype(fold_tag)::value;
            float ls0 = 0.f, ls1 = 0.f;
  #pragma unroll
            for (int k = 0; k < 8; ++k) {       // 16-byte chunk k holds columns 16k .. 16k+15
              const float cgk = cg[k >> 1];
              const float offk = kF4 ? goff[k >> 1] : negm;
              uint32_t wds[4];
              float fk[kFold ? 16 : 1];
              if constexpr (kFold) {
                const float4* cf = reinterpret_cast<const float4*>(vt + Lay::kVtColf) + 4 * k;
  #pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float4 f4 = cf[u];
                  fk[4 * u] = f4.x; fk[4 * u + 1] = f4.y; fk[4 * u + 2] = f4.z; fk[4 * u + 3] = f4.w;
                }
                if ((k >> 1) == dgrp) {
                  const uint4 vb = *reinterpret_cast<const uint4*>(vt + Lay::kVtBytesV + 16 * k);
                  const uint32_t vw[4] = {vb.x, vb.y, vb.z, vb.w};
  #pragma unroll
                  for (int u = 0; u < 16; ++u) {
                    // masked keys past the row may exceed the prefix maximum:
                    // their factor is capped at 1 (they multiply an exact 0)
                    const int e = min(static_cast<int>((vw[u >> 2] >> (8 * (u & 3))) & 0xffu) - sdiag - a.c_exp, 0);
                    fk[u] = e > -127 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : 0.f;
                  }
                }
              }
  #pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int c = 16 * k + 4 * q;
                float a0, a1, a2, a3;
                ffma2(a0, a1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), cgk, cgk, offk, offk);
                ffma2(a2, a3, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]), cgk, cgk, offk, offk);
                float p0 = ex2_approx(a0), p1 = ex2_approx(a1), p2 = ex2_approx(a2), p3 = ex2_approx(a3);
                fadd2(ls0, ls1, p0, p1);
                fadd2(ls0, ls1, p2, p3);
                if constexpr (kFold) {
                  fmul2(p0, p1, p0, p1, fk[4 * q], fk[4 * q + 1]);
                  fmul2(p2, p3, p2, p3, fk[4 * q + 2], fk[4 * q + 3]);
                }
                wds[q] = cvt_e4m3x4(p0, p1, p2, p3);
              }
              *reinterpret_cast<uint4*>(sP + rbase + ((k ^ (row & 7)) << 4)) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
              if constexpr (kF4) {
                if (k & 1) {                     // end of a 32-key group
                  lsum = fmaf(ls0 + ls1, gsc[k >> 1], lsum);
                  ls0 = ls1 = 0.f;
                }
              }
            }
            if constexpr (!kF4) lsum = ls0 + ls1;
          };
          if constexpr (kExact) {
            if (vfold) prob_loop(std::true_type{});
            else prob_loop(std::false_type{});
          } else {
            prob_loop(std::false_type{});
          }
        }
        l16 += lsum;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[Lay::bPFull + b]);
        if (j == 0 && pend.on) {
          if (!epilogue(pend)) { ok = false; break; }
          pend.on = false;
        }
      }
      if (!ok) { *abort_flag = 1; break; }
      pend = Pending{t, m, l16, w.h, it - 1, true, valid};
    }
    // the last item's epilogue
    if (pend.on && !*abort_flag && !epilogue(pend)) *abort_flag = 1;
    // every O store has landed before the CTA exits
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  } else {
    if constexpr (D == 64) setmaxnreg_dec<Lay::kRegsService>();
  }
  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    int it = 0, items = 0, q_issued = 0;
    ItemFeed feed{ring, a.plan_items, a.item_counter, total, a.Hq, a.schedule == 0,
                  SnakeIter{0, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total}, 0, 0, a.status, role_sleeps(kSleepMask, kRoleProducer)};
    int4 rec;
    int g = feed.next(rec);
    bool ok = feed.publish(g, rec);
    while (ok && g >= 0 && !*abort_flag) {
      const FwdItem w = decode_fwd(a, g, rec);
      // item k uses Q buffer k & 1, last used by item k - 2
      const int qb = items & 1;
      if (items >= 2 && !mbar_wait(&bars[Lay::bQEmpty + qb], ((items >> 1) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleProducer))) { ok = false; break; }
      if constexpr (kF4) {
        // the 4-bit S MMA's Q scale words for this Q buffer: per 64-element
        // chunk c, row r, word i = the four UE4M3 bytes of tile row 32 i + r
        const int64_t r0 = w.s_doc + w.qt * kTile;
#pragma unroll
        for (int c = 0; c < Lay::kC4; ++c) {
          uint32_t wq[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t tt = r0 + 32 * i + lane;
            wq[i] = tt < T ? __ldg(reinterpret_cast<const uint32_t*>(a.q4_scales + (tt * a.Hq + w.h) * (D / 16)) + c) : 0u;
          }
          reinterpret_cast<uint4*>(smem + Lay::kSq4 + (qb * Lay::kC4 + c) * 512)[lane] =
              make_uint4(wq[0], wq[1], wq[2], wq[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        const int32_t y = static_cast<int32_t>(w.s_doc + w.qt * kTile);
        if constexpr (kF4) {
          mbar_arrive_expect_tx(&bars[Lay::bQFull + qb], Lay::kTileBytes / 2);
          tma_load_2d(smem + Lay::kQ + qb * Lay::kTileBytes, &a.tm_q4, w.h * (D / 2), y, &bars[Lay::bQFull + qb]);
        } else {
          mbar_arrive_expect_tx(&bars[Lay::bQFull + qb], Lay::kTileBytes);
          tma_load_2d(smem + Lay::kQ + qb * Lay::kTileBytes, &a.tm_q, w.h * D, y, &bars[Lay::bQFull + qb]);
        }
      }
      ++q_issued;
      for (int j = 0; j < w.n_kt; ++j) {
        const int kt = fwd_key_tile(w, j, a.causal);
        const int st = it % Lay::kStages;
        if (it >= Lay::kStages &&
            !mbar_wait(&bars[Lay::bKVEmpty + st], ((it / Lay::kStages) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleProducer))) {
          ok = false;
          break;
        }
        // V block-scale word: byte g = UE8M0 scale of the 32-key group g of this tile
        uint32_t word = 0;
        // exact options: V's per-key exponent is folded into P-hat on the
        // diagonal tile of a causal call only (its blocks hold keys the early
        // rows do not see); the tiles before it take V's token-block codes
        const bool vfold = kExact && a.causal && kt == w.qt;
        if constexpr (kExact) {
          const uint8_t* ksc = a.k_scales + static_cast<int64_t>(w.hk) * T + w.s_doc;
          const int kbase = kt * kTile;
          // S MMA scale words of K: row r, word i = the scale byte of key 32 i + r
          uint32_t kw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rel = kbase + 32 * i + lane;
            kw[i] = (rel < w.L ? static_cast<uint32_t>(__ldg(ksc + rel)) : 127u) * 0x01010101u;
          }
          reinterpret_cast<uint4*>(smem + Lay::kSkb + st * 512)[lane] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
        }
        if (vfold) {
          // V's exponents are folded into P-hat: V's codes enter with scale 1
          word = 0x7f7f7f7fu;
          const uint8_t* vsc = a.v_scales + static_cast<int64_t>(w.hk) * T + w.s_doc;
          const int kbase = kt * kTile;
          // fold table: lane owns keys 4 lane .. 4 lane + 3 (group lane >> 3);
          // keys past the document end count as byte 0 and get factor 0
          uint32_t vb[4], lp[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int rel = kbase + 4 * lane + u;
            vb[u] = rel < w.L ? static_cast<uint32_t>(__ldg(vsc + rel)) : 0u;
            lp[u] = u == 0 ? vb[0] : max(lp[u - 1], vb[u]);
          }
          // inclusive scan of the lane maxima over the 8 lanes of a group
          uint32_t run = lp[3];
#pragma unroll
          for (int off = 1; off < 8; off <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, run, off, 8);
            if ((lane & 7) >= off) run = max(run, t);
          }
          uint32_t excl = __shfl_up_sync(0xffffffffu, run, 1, 8);
          if ((lane & 7) == 0) excl = 0;
          const uint32_t gmax = __shfl_sync(0xffffffffu, run, lane | 7);
          const int sg = max(static_cast<int>(gmax) - a.c_exp, 0);
          float fv[4];
          uint32_t pmw = 0, vbw = 0;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = static_cast<int>(vb[u]) - sg - a.c_exp;      // <= 0
            fv[u] = (kbase + 4 * lane + u < w.L && e > -127) ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : 0.f;
            pmw |= max(excl, lp[u]) << (8 * u);
            vbw |= vb[u] << (8 * u);
          }
          uint8_t* vt = smem + Lay::kVt + st * Lay::kVtBytes;
          reinterpret_cast<float4*>(vt + Lay::kVtColf)[lane] = make_float4(fv[0], fv[1], fv[2], fv[3]);
          reinterpret_cast<uint32_t*>(vt + Lay::kVtBytesV)[lane] = vbw;
          reinterpret_cast<uint32_t*>(vt + Lay::kVtPm)[lane] = pmw;
          const uint32_t s0 = __shfl_sync(0xffffffffu, sg, 0), s1 = __shfl_sync(0xffffffffu, sg, 8);
          const uint32_t s2 = __shfl_sync(0xffffffffu, sg, 16), s3 = __shfl_sync(0xffffffffu, sg, 24);
          if (lane == 0) *reinterpret_cast<uint32_t*>(vt + Lay::kVtPword) = s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
        } else {
          // token-block V scales (the exact options keep a token-block copy)
          const uint8_t* vsc = kExact ? a.vb_scales : a.v_scales;
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            const int rel = kt * kTile + gg * kBlock;
            const uint32_t byte = rel < w.L ? __ldg(vsc + static_cast<int64_t>(w.hk) * T + w.s_doc + rel) : 127u;
            word |= byte << (8 * gg);
          }
        }
        reinterpret_cast<uint4*>(smem + Lay::kSfb + st * 512)[lane] = make_uint4(word, word, word, word);
        if constexpr (kF4) {
          // the 4-bit S MMA's K scale words of this stage (same layout as Q's)
          const int64_t k0 = w.s_doc + kt * kTile;
#pragma unroll
          for (int c = 0; c < Lay::kC4; ++c) {
            uint32_t wk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int64_t tt = k0 + 32 * i + lane;
              wk[i] = tt < T ? __ldg(reinterpret_cast<const uint32_t*>(a.k4_scales + (tt * a.Hkv + w.hk) * (D / 16)) + c) : 0u;
            }
            reinterpret_cast<uint4*>(smem + Lay::kSk4 + (st * Lay::kC4 + c) * 512)[lane] =
                make_uint4(wk[0], wk[1], wk[2], wk[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int32_t y = static_cast<int32_t>(w.s_doc + kt * kTile);
          if constexpr (kF4) {
            mbar_arrive_expect_tx(&bars[Lay::bKVFull + st], Lay::kTileBytes / 2 + Lay::kTileBytes);
            tma_load_2d(smem + Lay::kK + st * Lay::kTileBytes, &a.tm_k4, w.hk * (D / 2), y, &bars[Lay::bKVFull + st]);
          } else {
            mbar_arrive_expect_tx(&bars[Lay::bKVFull + st], 2 * Lay::kTileBytes);
            tma_load_2d(smem + Lay::kK + st * Lay::kTileBytes, &a.tm_k, w.hk * D, y, &bars[Lay::bKVFull + st]);
          }
          tma_load_2d(smem + Lay::kV + st * Lay::kTileBytes, (kExact && !vfold) ? &a.tm_vb : &a.tm_v, w.hk * D, y,
                      &bars[Lay::bKVFull + st]);
        }
        __syncwarp();
        ++it;
      }
      if (!ok) break;
      ++items;
      // diagnostic: hand out no further item (not even the end marker)
      if (a.debug_item_limit > 0 && items >= a.debug_item_limit) break;
      // the next item is claimed once this one's last K/V loads are issued
      g = feed.next(rec);
      ok = feed.publish(g, rec);
    }
    if (!ok) *abort_flag = 1;
    // Let every copy still in flight land before the CTA can exit, also when
    // the loop ended because another warp gave up: the last phase armed on
    // each K/V stage and Q buffer (already complete after a normal run).
    for (int x = (it > Lay::kStages ? it - Lay::kStages : 0); x < it; ++x)
      mbar_wait(&bars[Lay::bKVFull + (x % Lay::kStages)], (x / Lay::kStages) & 1, nullptr);
    for (int x = (q_issued > 2 ? q_issued - 2 : 0); x < q_issued; ++x)
      mbar_wait(&bars[Lay::bQFull + (x & 1)], (x >> 1) & 1, nullptr);
  } else if (warp == 7) {
    // ------------------------------------------------------------ dQ accumulator clearing
    // Warp 7 takes every item from the ring (its release is counted by the
    // ring's empty barriers) and, at d = 64 with an accumulator, clears it.
    const bool clear = Lay::kZeroBytes > 0 && a.dqacc != nullptr;
    uint4* z = reinterpret_cast<uint4*>(smem + Lay::kZero);
    if (clear) {
      for (int i = lane; i < Lay::kZeroBytes / 16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) {
      work.whole_warp = false;
      work.sleep = role_sleeps(kSleepMask, kRoleDrain);
      for (;;) {
        int g;
        int4 rec;
        if (!work.next(g, rec) || *abort_flag) break;
        if (!clear) continue;
        const FwdItem w = decode_fwd(a, g, rec);
        // rows [s_doc + 128 qt, +128) of head h: 4 x 2 boxes of 32 rows x
        // 32 columns; rows past T are clipped, rows of the next document
        // are zeroed as well (they need it too)
        const int32_t y0 = static_cast<int32_t>(w.s_doc + w.qt * kTile);
#pragma unroll
        for (int rb = 0; rb < 4; ++rb) {
          tma_store_2d(&a.tm_dqz, w.h * D, y0 + 32 * rb, z);
          tma_store_2d(&a.tm_dqz, w.h * D + 32, y0 + 32 * rb, z);
        }
        bulk_commit_group();
        bulk_wait_group_read<4>();                 // bounded in-flight stores
      }
      if (clear) bulk_wait_group<0>();             // every store done before the CTA exits
    }
    __syncwarp();
  } else if (warp == 5 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 5 issues S = Q K^T, warp 6 O += P-hat V: neither chain waits
    // behind the other's blocked issue.  Each thread's commits track only its
    // own MMAs.
    if (lane == 0) {
      work.whole_warp = false;
      work.sleep = role_sleeps(kSleepMask, kRoleIssuer);
      int it = 0, items = 0;
      bool ok = true;
      if (warp == 5) {
        const uint32_t idesc_s = idesc_f8(128, 128, false, false);
        uint32_t sQ = smem_u32(smem + Lay::kQ);
        int qbuf = 0;                  // Q buffer of the current item (its scale-factor set)
        if constexpr (kExact) {
          // Q's scale 1 for every row (its exponent is in the softmax's row factor)
          uint4* sqa = reinterpret_cast<uint4*>(smem + Lay::kSqa);
          for (int i = 0; i < 32; ++i) sqa[i] = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
          fence_proxy_async_smem();
          tmem_cp_32x128b_x4(tbase + Lay::kTSqa, make_smem_desc(smem_u32(sqa), 0, 128, kSwizzleNone));
        }
        auto issue_s = [&](int x) -> bool {
          const int st = x % Lay::kStages;
          if (!mbar_wait(&bars[Lay::bKVFull + st], (x / Lay::kStages) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) return false;
          const int b = Lay::kSBufs == 2 ? (x & 1) : 0;
          if (x >= Lay::kSBufs && !mbar_wait(&bars[Lay::bSEmpty + b], ((x / Lay::kSBufs) - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) return false;
          tc_fence_after();
          const uint32_t sK = smem_u32(smem + Lay::kK + st * Lay::kTileBytes);
          if constexpr (kF4) {
            // NVFP4 path: 4-bit S MMA, K = 64 per instruction.  The stage's K
            // scale columns were last read by S(x - 3), complete since the
            // softmax released S(x - 1) or S(x - 2).
            constexpr uint32_t kSwz4 = D == 64 ? kSwizzle32B : kSwizzle64B;
#pragma unroll
            for (int c = 0; c < Lay::kC4; ++c)
              tmem_cp_32x128b_x4(tbase + Lay::kTSk4 + (st * Lay::kC4 + c) * 4,
                                 make_smem_desc(smem_u32(smem + Lay::kSk4 + (st * Lay::kC4 + c) * 512), 0, 128, kSwizzleNone));
#pragma unroll
            for (int c = 0; c < Lay::kC4; ++c) {
              const uint64_t ad = make_smem_desc(sQ + 32 * c, 16, 8 * (D / 2), kSwz4);
              const uint64_t bd = make_smem_desc(sK + 32 * c, 16, 8 * (D / 2), kSwz4);
              mma_mxf4nvf4(tbase + Lay::kTS + b * 128, ad, bd, idesc_mxf4nvf4(128, 128),
                           tbase + Lay::kTSq4 + (qbuf * Lay::kC4 + c) * 4, tbase + Lay::kTSk4 + (st * Lay::kC4 + c) * 4,
                           c > 0 ? 1u : 0u);
            }
          } else if constexpr (kExact) {
            // per-key K scales (exact options) applied by a block-scaled MMA;
            // this stage's columns were last read by S(x - 3), complete
            // since the softmax released S(x - 1)
            const uint32_t tkb = tbase + Lay::kTSkb + 4 * st;
            tmem_cp_32x128b_x4(tkb, make_smem_desc(smem_u32(smem + Lay::kSkb + st * 512), 0, 128, kSwizzleNone));
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              const uint64_t ad = make_smem_desc(sQ + 32 * kk, 16, 8 * D, Lay::kSwz);
              const uint64_t bd = make_smem_desc(sK + 32 * kk, 16, 8 * D, Lay::kSwz);
              mma_mxf8(tbase + Lay::kTS + b * 128, ad, bd, idesc_mxf8(128, 128, false, false, kk, kk),
                       tbase + Lay::kTSqa, tkb, kk > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              const uint64_t ad = make_smem_desc(sQ + 32 * kk, 16, 8 * D, Lay::kSwz);
              const uint64_t bd = make_smem_desc(sK + 32 * kk, 16, 8 * D, Lay::kSwz);
              mma_f8(tbase + Lay::kTS + b * 128, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&bars[Lay::bSFull + b]);
          return true;
        };
        for (;;) {
          int g;
          int4 rec;
          if (!work.next(g, rec) || *abort_flag) break;
          const FwdItem w = decode_fwd(a, g, rec);
          const int qb = items & 1;
          sQ = smem_u32(smem + Lay::kQ + qb * Lay::kTileBytes);
          qbuf = qb;
          if (!mbar_wait(&bars[Lay::bQFull + qb], (items >> 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
          tc_fence_after();
          if constexpr (kF4) {
            // this Q buffer's scale columns were last read by item (items - 2),
            // whose S MMAs completed before its Q buffer was released
#pragma unroll
            for (int c = 0; c < Lay::kC4; ++c)
              tmem_cp_32x128b_x4(tbase + Lay::kTSq4 + (qb * Lay::kC4 + c) * 4,
                                 make_smem_desc(smem_u32(smem + Lay::kSq4 + (qb * Lay::kC4 + c) * 512), 0, 128, kSwizzleNone));
          }
          for (int j = 0; j < w.n_kt; ++j) {
            if (!issue_s(it + j)) { ok = false; break; }
          }
          if (!ok) break;
          mma_commit(&bars[Lay::bQEmpty + qb]);         // Q is read by S only
          it += w.n_kt;
          ++items;
        }
      } else {
        const uint32_t pbyte = static_cast<uint32_t>(127 - a.c_exp);
        const uint32_t pword = pbyte | (pbyte << 8) | (pbyte << 16) | (pbyte << 24);
        uint32_t* sfa = reinterpret_cast<uint32_t*>(smem + Lay::kSfa);
        for (int i = 0; i < 128; ++i) sfa[i] = pword;
        fence_proxy_async_smem();
        tmem_cp_32x128b_x4(tbase + Lay::kTSfa, make_smem_desc(smem_u32(sfa), 0, 128, kSwizzleNone));
        const uint32_t sP = smem_u32(smem + Lay::kP);
        for (;;) {
          int g;
          int4 rec;
          if (!work.next(g, rec) || *abort_flag) break;
          const FwdItem w = decode_fwd(a, g, rec);
          for (int j = 0; j < w.n_kt; ++j) {
            const int x = it + j;
            const int pb = x & 1;
            // P-hat(x) written (so S(x) completed and K/V of this stage
            // landed); the first PV of an item overwrites O, which the
            // previous item's epilogue must have read.  The V scale columns
            // of this stage were last read by PV(x - 3), complete because the
            // softmax waited for PV(x - 2) before writing P-hat(x).
            if (!mbar_wait(&bars[Lay::bPFull + pb], (x >> 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) { ok = false; break; }
            if (j == 0 && items > 0 && !mbar_wait(&bars[Lay::bOEmpty], (items - 1) & 1, a.status, role_sleeps(kSleepMask, kRoleIssuer))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int st = x % Lay::kStages;
            const uint32_t sfb_t = tbase + Lay::kTSfb + 4 * st;
            tmem_cp_32x128b_x4(sfb_t, make_smem_desc(smem_u32(smem + Lay::kSfb + st * 512), 0, 128, kSwizzleNone));
            // exact options: P-hat's scale words, one per query row, written
            // by the softmax; buffer pb's columns were last read by PV(x - 2)
            uint32_t sfa_t = tbase + Lay::kTSfa;
            // exact options: per-row words on the diagonal tile (the V fold)
            // only; the tiles before it use the constant 2^-c
            const bool rowwords = kF4 || (kExact && a.causal && fwd_key_tile(w, j, a.causal) == w.qt);
            if constexpr (kExact || kF4) {
              if (rowwords) {
                sfa_t += (kExact ? 4 : 0) + 4 * pb;
                tmem_cp_32x128b_x4(sfa_t, make_smem_desc(smem_u32(smem + Lay::kPsw + pb * 512), 0, 128, kSwizzleNone));
              }
            }
            const uint32_t sV = smem_u32(smem + Lay::kV + st * Lay::kTileBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = make_smem_desc(sP + pb * (kTile * kTile) + 32 * kk, 16, 1024, kSwizzle128B);
              const uint64_t bd = make_smem_desc(sV + kk * 32 * D, 16, 8 * D, Lay::kSwz);
              const uint32_t id = idesc_mxf8(128, D, false, true, kk, kk);
              mma_mxf8(tbase + Lay::kTO, ad, bd, id, sfa_t, sfb_t, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars[Lay::bPVDone + pb]);
            // K (read by S(x), complete before P-hat(x)) and V of this stage
            mma_commit(&bars[Lay::bKVEmpty + st]);
          }
          if (!ok) break;
          it += w.n_kt;
          ++items;
        }
      }
      if (!ok) *abort_flag = 1;
      // every MMA this thread issued must be complete before TMEM is freed
      uint64_t* fin = &bars[warp == 5 ? Lay::bFinal : Lay::bFinal2];
      mma_commit(fin);
      mbar_wait(fin, 0, nullptr);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tbase, Lay::kTmemCols);
  // A forward that did not clear its items' dQ accumulator rows (it gave up,
  // or the plan was invalid) withdraws the stamp the quantize launch wrote,
  // so the backward clears the accumulator itself.
  if (threadIdx.x == 0 && a.dq_tag != nullptr && (*abort_flag || !valid_plan)) *a.dq_tag = 0;
}

template <int D, bool kExact, bool kDump = false, bool kF4 = false>
static void launch_fwd_t(const FwdArgs& a, int num_ctas, cudaStream_t st) {
  using Lay = FwdLayout<D, kExact, kF4>;
  constexpr int smem = Lay::kSmemAlloc;
  static std::atomic<uint64_t> configured{0};
  if (first_use_on_device(configured))
    cudaFuncSetAttribute(fwd_kernel<D, kExact, kDump, kF4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  fwd_kernel<D, kExact, kDump, kF4><<<num_ctas * Lay::kCtasPerSm, Lay::kThreads, smem, st>>>(a);
}

cudaError_t launch_fwd(const FwdArgs& a, int d, int num_ctas, cudaStream_t st) {
  if (a.dump.s != nullptr) {
    // diagnostic score-tile dump (token-block scales only)
    if (a.exact || a.nvfp4) return cudaErrorInvalidValue;
    if (d == 64) launch_fwd_t<64, false, true>(a, num_ctas, st);
    else launch_fwd_t<128, false, true>(a, num_ctas, st);
    return cudaGetLastError();
  }
  if (a.nvfp4) {
    if (d == 64) launch_fwd_t<64, false, false, true>(a, num_ctas, st);
    else launch_fwd_t<128, false, false, true>(a, num_ctas, st);
    return cudaGetLastError();
  }
  if (d == 64) {
    if (a.exact) launch_fwd_t<64, true>(a, num_ctas, st);
    else launch_fwd_t<64, false>(a, num_ctas, st);
  } else {
    if (a.exact) launch_fwd_t<128, true>(a, num_ctas, st);
    else launch_fwd_t<128, false>(a, num_ctas, st);
  }
  return cudaGetLastError();
}

}  // namespace flamia
