// Fused up-projection and absorb for decode (MlaPrologV2 README, 功能说明: q^C = c^Q·W^UQ,
// q^R = ROPE(c^Q·W^QR), q^N = q^C·W^UK), one CTA per head n, tokens as the MMA's M = 128 rows:
//
//   1. [q^C_n | q_r,n] = c^Q · [W^UQ_n | W^QR_n]   K = Hcq, N = D + Dr = 192 columns in TMEM
//   2. epilogue: q^C_n rounded to bf16 into shared memory, laid out as the next MMA's A operand;
//      q_r,n rotated (half-and-half RoPE of aclnnQkvRmsNormRopeCache "Formulas" (3)) -> query_rope
//   3. q^N_n = q^C_n · W^UK_n                         K = D, N = Hckv (chunks of 192 columns)
//   4. epilogue: q^N_n rounded to bf16 -> query
//
// q^C never leaves the SM, and the head's W^UK tiles stream through the same pipeline right
// behind its W^UQ|W^QR tiles, so one launch replaces two kernels and their boundary.  Weights are
// prepacked K-major: W^UQ|W^QR rows [all heads' nope rows n*D + d | all heads' rope rows, pairs
// (j, j + Dr/2) adjacent], W^UK as (N, Hckv, D).
//
// Each SM streams its weights at a bounded rate (about 40 GB/s on GB300 however they are
// fetched), so the SMs without a head take W^QR work: the rope rows come in 2N blocks of 32
// (block g = head g/2, pairs 16*(g%2)..+15).  With R such "rope CTAs" (blockIdx >= N), a head CTA
// keeps k of its own blocks (2, 1 or 0) and the rope CTAs share the others evenly, at most 6
// blocks (192 rows) each; a rope CTA runs only the up-projection and RoPE.
//
// Roles: warp 0 lane 0 TMA producer, warp 1 lane 0 MMA issuer, warp 2 TMEM owner, warps 4..7
// epilogue (warp 4 + q owns TMEM lanes 32q..32q+31, i.e. tokens 32q..32q+31).  With an int8
// W^UQ|W^QR (partial and full quant) warp 3 lane 0 loads the raw int8 tiles into a ring of
// their own (starting before the preceding kernel completes), warps 8..11 expand each into the
// f16 operand layout (exact; the c^Q codes are f16 too), and the epilogue dequantises
// acc * scale_t[t] * dequant_scale_w_uq_qr[col] (the CTA's columns of the scales staged in
// shared memory while the up-projection runs) before q^C is rounded and q_r rotated.  The
// epilogue releases q^C to the absorb MMAs before it rotates the rope blocks.  c^Q tiles carry
// the token rows only (T rounded up to 8); the MMA's other A rows feed accumulator lanes that
// are never stored.  Every mbarrier wait is bounded; on a timeout the CTA lets its issued
// loads land, frees TMEM and latches the error word.
//
// Head pairs (2N <= SMs): a head's work is split over the two CTAs of a cluster.  CTA r of the
// pair computes q^C columns 64r..64r+63 (its 64 W^UQ rows, plus the head's rope block r), sends
// that 64-wide K block of the absorb's A operand to the other CTA's shared memory with one bulk
// copy per epilogue warp, and computes q^N for its half of the Hckv columns from both K blocks.
// Each CTA then streams about half of a head's W^UQ and W^UK bytes, where with N heads on one
// CTA each the N head CTAs carry most of the bytes and the remaining SMs little.
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "internal.h"

namespace mlap {

namespace {

constexpr int kUaBK = 64;                              // K elements per stage
constexpr int kUaA = 128 * kUaBK * 2;                  // c^Q tile: 128 tokens x 64 (16 KB)
constexpr int kUaBars = 1024;                          // barriers and flags, ahead of the stages
constexpr int kUaDqFloats = 192;                       // int8: staged dequant scales, after them
static_assert(kUaDqFloats * 4 <= kUaBars, "the dequant scales of up to 192 weight rows");
constexpr int kUaSmemMax = 232448;                     // 227 KB opt-in per CTA
constexpr int kUaMaxStages = 8;

// Shared memory (after 1024-B alignment): barriers, then the operand stages (c^Q tile + weight
// tile), each holding exactly this CTA's weight rows (a head CTA 128 + 32k, a rope CTA 32 per
// block), so a head CTA with one rope block fits six 36 KB stages where fixed 40 KB stages fit
// four: more of the weight stream in flight, which is what the per-SM rate depends on.  q^C
// lives in the c^Q halves of stages 0 and 1 once the up-projection is done.  int8 weight: after
// the operand stages, a ring of raw int8 tiles (64 B per row), filled by a second producer thread
// so that more of the weight stream is in flight than there are operand stages; up to six raw
// tiles, as many as leave room for four operand stages.
template <bool INT8>
struct UaCfg {
  static constexpr int THREADS = INT8 ? 384 : 256;
  static constexpr int MAX_RAW = INT8 ? 6 : 0;
  static constexpr int SMEM = kUaSmemMax;
};
constexpr uint32_t kUaUpCol = 256;                     // TMEM column of the up accumulator
// Operand stages whose weight tiles the producer requests before its wait on the preceding
// kernel (six were slower: their loads queue ahead of the preceding kernels' own in DRAM).
constexpr int kUaPreStages = 4;
constexpr int kD = 128;
constexpr int kDr = 64;

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}

__device__ __forceinline__ void unpack16(uint4 a, uint4 b, float* out) {
  const __nv_bfloat16* ea = reinterpret_cast<const __nv_bfloat16*>(&a);
  const __nv_bfloat16* eb = reinterpret_cast<const __nv_bfloat16*>(&b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    out[i] = __bfloat162float(ea[i]);
    out[8 + i] = __bfloat162float(eb[i]);
  }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// This CTA's share: head CTA (blockIdx < N) or rope CTA, and its rope blocks g_j = g0 + gs * j,
// j < nrope (kept in registers: the producer's issue path is latency-critical).
// A head CTA of a pair also has its head n and its rank r in the pair.
struct UaPlan {
  bool head;
  int nrope, g0, gs;
  int n, r;
};

template <bool PAIR>
__device__ __forceinline__ UaPlan ua_plan(const UpAbsorbParams& p) {
  UaPlan pl;
  const int b = blockIdx.x;
  const int nhc = PAIR ? 2 * p.N : p.N;                // head CTAs
  pl.n = PAIR ? b >> 1 : b;
  pl.r = PAIR ? b & 1 : 0;
  if (b < nhc) {   // (with k = 1 the CTA of rank r in a pair takes the head's rope block r)
    pl.head = true;
    pl.nrope = p.k;
    pl.g0 = PAIR ? b : 2 * b;
    pl.gs = 1;
  } else {
    const int r = b - nhc;
    const int total = p.k == 1 ? (PAIR ? 0 : p.N) : 2 * p.N;   // blocks the rope CTAs share
    const int i0 = static_cast<int>(static_cast<long long>(total) * r / p.R);
    const int i1 = static_cast<int>(static_cast<long long>(total) * (r + 1) / p.R);
    pl.head = false;
    pl.nrope = i1 - i0 < 6 ? i1 - i0 : 6;
    pl.g0 = p.k == 1 ? 2 * i0 + 1 : i0;
    pl.gs = p.k == 1 ? 2 : 1;
  }
  return pl;
}

// The int8 kernel's producers also take a head CTA's contiguous W^UQ rows (128, or the 64 of a
// pair CTA), and 128 W^UK rows, as one box each: at these sizes each TMA issue costs the
// producer thread about as much time as the box it moves.  The bf16 kernel is not
// producer-bound and takes no extra maps (two more tensor maps in its parameters cost its
// launch more than the larger boxes would save).
template <bool INT8> struct UaWideMaps {
  CUtensorMap w;    // W^UQ|W^QR rows, box 64 x 128 (64 x 64 for head pairs)
  CUtensorMap uk;   // W^UK rows, box 64 x 128
};
template <> struct UaWideMaps<false> {};

template <bool INT8, bool PAIR>
__global__ void __launch_bounds__(UaCfg<INT8>::THREADS, 1)
    up_absorb_kernel(const __grid_constant__ CUtensorMap tmCq,   // c^Q (T, Hcq), box 64 x 128
                     const __grid_constant__ CUtensorMap tmW,    // W^UQ|W^QR rows, box 64 x 32
                     const __grid_constant__ CUtensorMap tmUk,   // W^UK rows, box 64 x 32
                     const __grid_constant__ UaWideMaps<INT8> wide,
                     const UpAbsorbParams p, uint32_t* __restrict__ err_word) {
  using Cfg = UaCfg<INT8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const UaPlan pl = ua_plan<PAIR>(p);
  const int n = pl.n;                                  // head (head CTAs)
  const int kb_up = (p.Hcq + kUaBK - 1) / kUaBK;
  constexpr int kHRows = PAIR ? kD / 2 : kD;           // this CTA's W^UQ rows of its head
  const int hrow0 = n * kD + kHRows * pl.r;            // the first of them
  const int up_rows = (pl.head ? kHRows : 0) + 32 * pl.nrope;   // B rows of the up-projection
  // this CTA's q^N columns c_lo..c_lo+cspan-1 (a pair splits the 32-column groups)
  const int hA = PAIR ? (p.Hckv / 32 + 1) / 2 * 32 : p.Hckv;
  const int c_lo = pl.r * hA;
  const int cspan = pl.r == 0 ? hA : p.Hckv - hA;
  // weight rows one stage holds (also the W^UK chunk height of a head CTA), the stage size and
  // the stage count
  const int wrows = up_rows;
  const int kUaStage = kUaA + wrows * kUaBK * 2;
  // (int8: the CTA's dequant scales follow the barriers, in a second KB ahead of the stages)
  constexpr int kHead = INT8 ? 2 * kUaBars : kUaBars;
  constexpr int kAvail = kUaSmemMax - 1024 - kHead - (PAIR ? kUaA : 0);
  const int kRawB = INT8 ? wrows * kUaBK : 0;                 // raw int8 tile bytes
  const int kRS = INT8 ? ((kAvail - 4 * kUaStage) / kRawB < Cfg::MAX_RAW
                              ? (kAvail - 4 * kUaStage) / kRawB : Cfg::MAX_RAW)
                       : 0;
  const int kUaStages = (kAvail - kRS * kRawB) / kUaStage < kUaMaxStages
                            ? (kAvail - kRS * kRawB) / kUaStage : kUaMaxStages;
  const int nh = pl.head ? (cspan + wrows - 1) / wrows : 0;   // absorb column chunks (<= 4)
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty_bar = full_bar + kUaMaxStages;
  uint64_t* rawf_bar = empty_bar + kUaMaxStages;       // int8: raw weight tile landed
  uint64_t* rawe_bar = rawf_bar + kUaMaxStages;        // int8: raw tile converted, slot free
  uint64_t* up_bar = rawe_bar + kUaMaxStages;          // up accumulator complete
  uint64_t* qc_bar = up_bar + 1;                       // q^C in smem, its accumulator read
  uint64_t* ab_bar = qc_bar + 1;                       // absorb chunk h complete (h < 4)
  uint64_t* qcr_bar = ab_bar + 4;                      // pair: the other CTA's K block landed
  uint64_t* rp_bar = qcr_bar + 1;                      // rope columns of the accumulator read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rp_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* dq_s = reinterpret_cast<float*>(smem + kUaBars);   // int8: up_rows dequant scales
  uint8_t* stages = smem + kHead;
  uint8_t* ring_raw = stages + kUaStages * kUaStage;   // int8: raw weight tiles
  // q^C operand, two 64-wide K blocks: the c^Q halves of stages 0 and 1, free once the
  // up-projection's MMAs have completed.  A pair computes K block r in the c^Q half of stage 0
  // and receives the other one in a region of its own after the raw ring (the other CTA may
  // send it before this CTA's up-projection is done).
  uint8_t* qc0 = stages;
  uint8_t* qc1 = stages + kUaStage;
  uint8_t* qc_peer = ring_raw + kRS * kRawB;
  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_UP, kStampStart);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmCq);
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmUk);
    if constexpr (INT8) {
      prefetch_tmap(&wide.w);
      prefetch_tmap(&wide.uk);
    }
  }
  if (warp == 1 && lane == 0) {
    for (int i = 0; i < kUaStages; ++i) {
      mbar_init(&full_bar[i], INT8 ? 1 + 4 : 1);   // producer (+ the four converter warps)
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < kRS; ++i) {
      mbar_init(&rawf_bar[i], 1);
      mbar_init(&rawe_bar[i], 4);                   // the four converter warps
    }
    mbar_init(up_bar, 1);
    mbar_init(qc_bar, 4);
    mbar_init(rp_bar, 4);
    for (int h = 0; h < 4; ++h) mbar_init(&ab_bar[h], 1);
    if constexpr (PAIR) {   // completes when the other CTA's four copies (16 KB) have landed
      mbar_init(qcr_bar, 1);
      mbar_arrive_expect_tx(qcr_bar, kUaA);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();   // the other CTA's barrier exists before its copy targets it
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  grid_launch_dependents();
  const bool producer = warp == 0 && lane == 0;
  const bool raw_producer = INT8 && warp == 3 && lane == 0;   // int8 weight tiles only
  // Every role but the producers waits here for the preceding kernel.  The int8 raw producer's
  // whole warp skips the wait, so that it fills its ring before that kernel completes (a wait
  // taken by some lanes of a warp can hold the warp's other lanes as well).  The W^UQ|W^QR
  // producer requests its first weight stages, then waits itself; the other lanes of its warp
  // wait here (measured: the decode call is fastest so, 1.4 us faster than with the whole warp
  // skipping this wait and 2 us faster than with the producer waiting before its requests).
  if (!producer && !(INT8 && warp == 3)) grid_dependency_wait();

  if (producer) {
    // ------------------------------------------------------------------ TMA producer
    int fills[kUaMaxStages] = {};
    // head n's W^UQ rows (D, or this CTA's D/2 of a pair), then this CTA's rope blocks: up to
    // six 32-row boxes per tile, their first weight rows computed once
    const int nbox = up_rows / 32;
    int ybox[6];
#pragma unroll
    for (int j = 0; j < 6; ++j) {
      const int jr = pl.head ? j - kHRows / 32 : j;   // rope block index of box j
      ybox[j] = jr < 0 ? hrow0 + 32 * j : p.N * kD + 32 * (pl.g0 + pl.gs * jr);
    }
    auto issue_w = [&](int st, int kb) {
      if constexpr (!INT8) {   // (int8 weight tiles come from the raw producer)
        uint8_t* b = stages + st * kUaStage + kUaA;
        mbar_expect_tx(&full_bar[st], static_cast<uint32_t>(up_rows) * kUaBK * 2);
#pragma unroll
        for (int j = 0; j < 6; ++j)
          if (j < nbox) tma_load_2d(b + j * 4096, &tmW, &full_bar[st], kb * kUaBK, ybox[j]);
      }
    };
    int pre = kb_up < kUaStages ? kb_up : kUaStages;
    if (pre > kUaPreStages) pre = kUaPreStages;
    for (int i = 0; i < pre; ++i) issue_w(i, i);      // weights do not depend on earlier kernels
    grid_dependency_wait();
    stamp(p.stamps, MLAP_STAMP_UP, kStampDep);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int kb = 0; ok && kb < kb_up; ++kb) {
      if (kb >= pre) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        issue_w(stage, kb);
      }
      mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(p.cq_rows) * kUaBK * 2);
      tma_load_2d(stages + stage * kUaStage, &tmCq, &full_bar[stage], kb * kUaBK, 0);
      ++fills[stage];
      if (++stage == kUaStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // head n's W^UK rows c_lo.., chunk h of wrows rows, K block kb2 of D
    for (int h = 0; ok && h < nh; ++h) {
      const int rows = cspan - h * wrows < wrows ? cspan - h * wrows : wrows;
      for (int kb2 = 0; kb2 < kD / kUaBK; ++kb2) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* b = stages + stage * kUaStage + kUaA;
        mbar_arrive_expect_tx(&full_bar[stage], rows * kUaBK * 2);
        int r = 0;
        if constexpr (INT8)
          for (; r + 128 <= rows; r += 128)
            tma_load_2d(b + r * 128, &wide.uk, &full_bar[stage], kb2 * kUaBK,
                        n * p.Hckv + c_lo + h * wrows + r);
        for (; r < rows; r += 32)
          tma_load_2d(b + r * 128, &tmUk, &full_bar[stage], kb2 * kUaBK,
                      n * p.Hckv + c_lo + h * wrows + r);
        ++fills[stage];
        if (++stage == kUaStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (*abort_flag) {
      // let every issued load land before the CTA exits (the last fill of stage i has parity
      // (fills[i] - 1) & 1; prefetched weights count toward the fill of their k block)
      const uint64_t t0 = globaltimer_ns();
      for (int i = 0; i < kUaStages; ++i) {
        if (fills[i] == 0 && i >= pre) continue;
        const uint32_t par = static_cast<uint32_t>((fills[i] > 0 ? fills[i] : 1) - 1) & 1u;
        while (!mbar_try_wait(&full_bar[i], par) && globaltimer_ns() - t0 < 20000000ull) {
        }
      }
    }
  } else if (raw_producer) {
    // ------------------------------------------------------------------ int8 weight producer
    // raw int8 rows of 64 B into a ring of kRS tiles, ahead of the operand stages
    int rawfills[kUaMaxStages] = {};
    const int nbox = up_rows / 32;
    int ybox[6];
#pragma unroll
    for (int j = 0; j < 6; ++j) {
      const int jr = pl.head ? j - kHRows / 32 : j;
      ybox[j] = jr < 0 ? hrow0 + 32 * j : p.N * kD + 32 * (pl.g0 + pl.gs * jr);
    }
    int rs = 0;
    uint32_t rph = 0;
    for (int kb = 0; kb < kb_up; ++kb) {
      if (kb >= kRS && !mbar_wait(&rawe_bar[rs], rph ^ 1u, abort_flag)) break;
      uint8_t* r = ring_raw + rs * kRawB;
      mbar_arrive_expect_tx(&rawf_bar[rs], static_cast<uint32_t>(up_rows) * kUaBK);
      // a head CTA's contiguous W^UQ rows (128, or 64 in a pair) as one box
      if constexpr (INT8)
        if (pl.head) tma_load_2d(r, &wide.w, &rawf_bar[rs], kb * kUaBK, hrow0);
#pragma unroll
      for (int j = 0; j < 6; ++j)
        if (j < nbox && !(pl.head && j < kHRows / 32))
          tma_load_2d(r + j * 2048, &tmW, &rawf_bar[rs], kb * kUaBK, ybox[j]);
      ++rawfills[rs];
      if (++rs == kRS) {
        rs = 0;
        rph ^= 1u;
      }
    }
    if (*abort_flag) {   // let every issued raw tile land before the CTA exits
      const uint64_t t0 = globaltimer_ns();
      for (int i = 0; i < kRS; ++i) {
        if (rawfills[i] == 0) continue;
        const uint32_t par = static_cast<uint32_t>(rawfills[i] - 1) & 1u;
        while (!mbar_try_wait(&rawf_bar[i], par) && globaltimer_ns() - t0 < 20000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // (int8 weight: the converted tiles and the c^Q codes are f16; the absorb stays bf16)
      const uint32_t idesc_up = INT8 ? idesc_f16_f32(128, up_rows) : idesc_bf16_f32(128, up_rows);
      for (int kb = 0; kb < kb_up; ++kb) {
        if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a = smem_u32(stages + stage * kUaStage);
        const uint32_t b = a + kUaA;
#pragma unroll
        for (int kk = 0; kk < kUaBK / 16; ++kk)
          umma_bf16_ss(tmem_base + kUaUpCol, sdesc_kmajor_sw128(a + kk * 32),
                       sdesc_kmajor_sw128(b + kk * 32), idesc_up, (kb > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&empty_bar[stage]);
        if (++stage == kUaStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) umma_commit(up_bar);
      if (ok && pl.head) ok = mbar_wait(qc_bar, 0, abort_flag);   // q^C staged, acc read
      if constexpr (PAIR)   // the other CTA's K block (always awaited: it lands here regardless)
        if (ok && pl.head) ok = mbar_wait_cluster(qcr_bar, 0, abort_flag);
      if (ok && pl.head) {
        tc_fence_after_sync();
        uint32_t qa[2] = {smem_u32(qc0), smem_u32(qc1)};
        if constexpr (PAIR) {
          qa[pl.r] = smem_u32(qc0);
          qa[pl.r ^ 1] = smem_u32(qc_peer);
        }
        bool rope_read = false;
        for (int h = 0; ok && h < nh; ++h) {
          const int rows = cspan - h * wrows < wrows ? cspan - h * wrows : wrows;
          const uint32_t idesc_ab = idesc_bf16_f32(128, rows);
          // a chunk whose accumulator columns reach the up accumulator's rope columns waits for
          // the epilogue to have read them (the q^C columns were read before qc_bar)
          if (!rope_read && h * wrows + rows > static_cast<int>(kUaUpCol) + kHRows) {
            ok = mbar_wait(rp_bar, 0, abort_flag);
            rope_read = true;
            tc_fence_after_sync();
            if (!ok) break;
          }
          for (int kb2 = 0; kb2 < kD / kUaBK; ++kb2) {
            if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t b = smem_u32(stages + stage * kUaStage) + kUaA;
#pragma unroll
            for (int kk = 0; kk < kUaBK / 16; ++kk)
              umma_bf16_ss(tmem_base + static_cast<uint32_t>(h * wrows),
                           sdesc_kmajor_sw128(qa[kb2] + kk * 32),
                           sdesc_kmajor_sw128(b + kk * 32), idesc_ab,
                           (kb2 > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&empty_bar[stage]);
            if (++stage == kUaStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) umma_commit(&ab_bar[h]);   // its stores overlap the next chunk's W^UK loads
        }
      }
    }
  } else if (INT8 && warp >= 8) {
    // ------------------------------------------------------------------ int8 -> bf16 converters
    const int ct = threadIdx.x - 256;
    int stage = 0, rs = 0;
    uint32_t phase = 0, rph = 0;
    bool ok = true;
    for (int kb = 0; kb < kb_up; ++kb) {
      // the raw tile has landed and the operand stage's previous round has been consumed
      if (!mbar_wait(&rawf_bar[rs], rph, abort_flag) ||
          !mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* raw = ring_raw + rs * kRawB;
      uint8_t* dst = stages + stage * kUaStage + kUaA;
      convert_int8_tile<6>(raw, dst, up_rows, ct);     // (up_rows <= 192)
      fence_proxy_async_shared();                      // generic writes -> the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&full_bar[stage]);
        mbar_arrive(&rawe_bar[rs]);                    // raw slot free for the producer
      }
      if (++stage == kUaStages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++rs == kRS) {
        rs = 0;
        rph ^= 1u;
      }
    }
    // the W^UK tiles are bf16: each converter warp only adds its arrival, once the stage's
    // previous round has been consumed (so that it cannot count toward that round)
    for (int i = 0; ok && i < nh * (kD / kUaBK); ++i) {
      if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_bar[stage]);
      if (++stage == kUaStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp - 4;
    const int t = q * 32 + lane;                       // token of this lane
    const bool live = t < p.T;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // RoPE tables of this token: pairs 0..15 and 16..31 at columns j and j + Dr/2
    uint4 cs[2][4], sn[2][4];
    if (live) {
      const uint4* c = reinterpret_cast<const uint4*>(p.cos + static_cast<size_t>(t) * kDr);
      const uint4* s = reinterpret_cast<const uint4*>(p.sin + static_cast<size_t>(t) * kDr);
#pragma unroll
      for (int i = 0; i < 4; ++i) {   // uint4 i covers columns 8i..8i+7
        cs[i >> 1][i & 1] = __ldg(c + i);
        sn[i >> 1][i & 1] = __ldg(s + i);
        cs[i >> 1][2 + (i & 1)] = __ldg(c + 4 + i);
        sn[i >> 1][2 + (i & 1)] = __ldg(s + 4 + i);
      }
    }
    // int8 weight: acc * scale_t[t] * dequant_scale_w_uq_qr[original column]; the CTA's
    // columns of dequant_scale_w_uq_qr go to shared memory while the up-projection runs
    const float st = INT8 && live ? __ldg(p.scale_t + t) : 0.f;
    if constexpr (INT8) {
      const int nq = pl.head ? kHRows : 0;
      for (int i = q * 32 + lane; i < up_rows; i += 128) {
        int c;
        if (i < nq) {        // nope row n*D + d is column n*(D+Dr) + d
          c = n * (kD + kDr) + kHRows * pl.r + i;
        } else {             // rope row i of head g/2 is column D + i/2 + (i%2)*Dr/2
          const int j = (i - nq) >> 5, ii = (i - nq) & 31;
          const int g = pl.g0 + pl.gs * j;
          c = (g >> 1) * (kD + kDr) + kD + (g & 1) * 16 + (ii >> 1) + (ii & 1) * (kDr / 2);
        }
        dq_s[i] = __ldg(p.dqw + c);
      }
      named_barrier_sync(1, 128);                      // the four epilogue warps
    }
    bool ok = mbar_wait(up_bar, 0, abort_flag);
    if (ok) {
      tc_fence_after_sync();
      if (q == 0 && lane == 0) stamp(p.stamps, MLAP_STAMP_UP, kStampMain);
      int col = 0;
      if (pl.head) {
        // q^C: bf16 into the K-major, 128B-swizzled A operand (token t = row t)
#pragma unroll 1
        for (; col < kHRows; col += 32) {
          float v[32];
          tmem_ld32(lane_base + kUaUpCol + col, v);
          if constexpr (INT8) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = v[j] * st * dq_s[col + j];
          }
          uint8_t* row = (PAIR || col < kUaBK ? qc0 : qc1) + t * 128;
          const int ch0 = (col % kUaBK) / 8;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(row + ((((ch0 + j) ^ (t & 7)) & 7) << 4)) = pack8(v + 8 * j);
        }
        // q^C is complete: the absorb may start while the rope blocks below are rotated
        tc_fence_before_sync();
        fence_proxy_async_shared();                    // q^C stores -> visible to the MMA
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)   // this warp's 32 rows (4 KB) of the K block -> the other CTA
            bulk_copy_to_peer(mapa_shared(smem_u32(qc_peer + q * 4096), pl.r ^ 1), qc0 + q * 4096,
                              4096, mapa_shared(smem_u32(qcr_bar), pl.r ^ 1));
          mbar_arrive(qc_bar);
        }
      }
      // rope blocks: 32 columns = pairs p0..p0+15 (p0 = 16 * (g % 2)) of head g / 2, RoPE,
      // -> query_rope
#pragma unroll 1
      for (int j = 0; j < pl.nrope; ++j, col += 32) {
        float y[32];
        tmem_ld32(lane_base + kUaUpCol + col, y);
        const int g = pl.g0 + pl.gs * j;
        const int half = g & 1;
        if constexpr (INT8) {
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = y[i] * st * dq_s[col + i];
        }
        if (live) {
          float c0[16], s0[16], c1[16], s1[16];
          unpack16(half ? cs[1][0] : cs[0][0], half ? cs[1][1] : cs[0][1], c0);
          unpack16(half ? sn[1][0] : sn[0][0], half ? sn[1][1] : sn[0][1], s0);
          unpack16(half ? cs[1][2] : cs[0][2], half ? cs[1][3] : cs[0][3], c1);
          unpack16(half ? sn[1][2] : sn[0][2], half ? sn[1][3] : sn[0][3], s1);
          float oa[16], ob[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float y0 = y[2 * i], y1 = y[2 * i + 1];
            oa[i] = y0 * c0[i] - y1 * s0[i];
            ob[i] = y1 * c1[i] + y0 * s1[i];
          }
          __nv_bfloat16* out =
              p.qr_out + (static_cast<size_t>(t) * p.N + (g >> 1)) * kDr + half * 16;
          uint4* da = reinterpret_cast<uint4*>(out);
          uint4* db = reinterpret_cast<uint4*>(out + kDr / 2);
          da[0] = pack8(oa);
          da[1] = pack8(oa + 8);
          db[0] = pack8(ob);
          db[1] = pack8(ob + 8);
        }
      }
      if (pl.head) {   // the rope columns have been read
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(rp_bar);
      }
    }
    if (ok && pl.head) {
      // query in groups of 64 columns: each lane (token) packs its 64 values into a 128-B row
      // of the warp's 4 KB staging tile (a c^Q half of a stage, free after the up-projection;
      // 16-B chunks XOR-swizzled by row), then eight lanes store each row as one 128-B line, four
      // rows per instruction, instead of 32 scattered 16-B pieces
      uint8_t* tile = stages + (2 + (q >> 1)) * kUaStage + (q & 1) * 4096;
      const int rsub = lane >> 3, ch = lane & 7;        // read-back: row rsub + 4i, chunk ch
      int waited = 0;                                   // absorb chunks known complete
#pragma unroll 1
      for (int c = 0; ok && c < cspan; c += 64) {
        const int w = cspan - c < 64 ? cspan - c : 64;     // 64, or 32 for the last group
        const int need = (c + w - 1) / wrows + 1;          // chunks holding columns c..c+w-1
        while (waited < need) {
          if (!mbar_wait(&ab_bar[waited], 0, abort_flag)) {
            ok = false;
            break;
          }
          ++waited;
        }
        if (!ok) break;
        tc_fence_after_sync();
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (g * 32 >= w) break;
          float v[32];
          tmem_ld32(lane_base + static_cast<uint32_t>(c + 32 * g), v);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(tile + lane * 128 + ((((4 * g + j) ^ (lane & 7)) & 7) << 4)) =
                pack8(v + 8 * j);
        }
        __syncwarp();
        if (ch * 8 < w) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = rsub + 4 * i;                 // token q*32 + r
            const int tr = q * 32 + r;
            const uint4 val =
                *reinterpret_cast<const uint4*>(tile + r * 128 + (((ch ^ (r & 7)) & 7) << 4));
            if (tr < p.T)
              *reinterpret_cast<uint4*>(p.q_out + (static_cast<size_t>(tr) * p.N + n) * p.Hckv +
                                        c_lo + c + ch * 8) = val;
          }
        }
        __syncwarp();                                   // the tile is read before it is rewritten
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) {
    // Neither CTA of a pair exits while a copy between them may still be in flight: after a
    // timeout, give copies issued so far time to land (bounded) on both sides of the pair's
    // final barrier, which each CTA reaches only after its own copy was issued or skipped.
    const bool aborted = *abort_flag != 0;
    if (aborted) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) {
      }
    }
    cluster_sync();
    if (aborted) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) {
      }
    }
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(err_word, kErrTimeout);
  if (threadIdx.x == 0) stamp(p.stamps, MLAP_STAMP_UP, kStampEnd);
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

void up_absorb_plan(int sms, int N, int* k, int* R, int* pair) {
  // Head pairs when two CTAs per head fit on the SMs: each CTA keeps one rope block, no rope
  // CTAs.  Otherwise rope blocks per head CTA (k) and rope CTAs (R) so that the CTAs stream
  // about the same weight bytes and a rope CTA takes at most 6 blocks.
  *pair = 2 * N <= sms ? 1 : 0;
  if (*pair) {
    *k = 1;
    *R = 0;
    return;
  }
  *R = sms - N;
  if (*R > 0 && 2 * N <= 6 * *R) {
    *k = 0;
    if (*R > 2 * N) *R = 2 * N;
  } else if (*R > 0 && N <= 6 * *R) {
    *k = 1;
    if (*R > N) *R = N;
  } else {
    *k = 2;
    *R = 0;
  }
}

bool up_absorb_supported(int64_t T, int64_t N, int64_t D, int64_t Dr, int64_t Hckv) {
  return T >= 1 && T <= 128 && N >= 1 && D == kD && Dr == kDr && Hckv >= 32 && Hckv <= 512 &&
         Hckv % 32 == 0;
}

template <bool INT8, bool PAIR>
static cudaError_t launch_ua_t(const CUtensorMap& tmCq, const CUtensorMap& tmW,
                               const CUtensorMap& tmUk, const UaWideMaps<INT8>& wide,
                               const UpAbsorbParams& p, uint32_t* err, cudaStream_t stream) {
  auto kern = up_absorb_kernel<INT8, PAIR>;
  constexpr int kSmem = UaCfg<INT8>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const int grid = (PAIR ? 2 * p.N : p.N) + p.R;
  if (PAIR && (grid & 1)) return cudaErrorInvalidValue;   // whole clusters of two
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(UaCfg<INT8>::THREADS);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, tmCq, tmW, tmUk, wide, p, err);
}

cudaError_t launch_up_absorb(const CUtensorMap& tmCq, const CUtensorMap& tmW,
                             const CUtensorMap& tmUk, const CUtensorMap* tmW128,
                             const CUtensorMap* tmUk128, const UpAbsorbParams& p, uint32_t* err,
                             cudaStream_t stream) {
  if ((tmW128 == nullptr) != (tmUk128 == nullptr)) return cudaErrorInvalidValue;
  if (p.cq_rows < 8 || p.cq_rows > 128 || p.cq_rows % 8 != 0 || p.cq_rows < (p.T < 128 ? p.T : 128))
    return cudaErrorInvalidValue;
  if (tmW128) {
    const UaWideMaps<true> wide{*tmW128, *tmUk128};
    return p.pair ? launch_ua_t<true, true>(tmCq, tmW, tmUk, wide, p, err, stream)
                  : launch_ua_t<true, false>(tmCq, tmW, tmUk, wide, p, err, stream);
  }
  return p.pair ? launch_ua_t<false, true>(tmCq, tmW, tmUk, UaWideMaps<false>{}, p, err, stream)
                : launch_ua_t<false, false>(tmCq, tmW, tmUk, UaWideMaps<false>{}, p, err, stream);
}

}  // namespace mlap
