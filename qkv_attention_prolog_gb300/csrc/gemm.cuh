// Persistent, warp-specialised tcgen05 GEMM used by every contraction of the MLA prolog.
//
//   C[m, n] = sum_k A[m, k] * B[n, k]      (both operands K-major bf16, fp32 accumulation)
//
// A and B arrive through TMA tensor maps (128-byte swizzle, 64-element K blocks).  A tile of
// BM=128 rows of A and BN rows of B is accumulated in tensor memory (TMEM) by one thread issuing
// tcgen05.mma; four epilogue warps read the accumulator back with tcgen05.ld, hand 32 x 32 blocks
// to an epilogue functor (the fused rounding, RoPE, dequant, ...) and write its output with TMA
// stores.  TMEM holds two accumulators so the epilogue of one tile overlaps the MMAs of the next.
//
// One operand is a weight (`w_op`).  Its first pipeline stages are requested before the kernel
// waits on the previous kernel in the stream (programmatic dependent launch), so the weight
// stream starts while the producer of the activations is still finishing.  With WQ != 0 the
// weight is int8: TMA brings the raw int8 tile and four converter warps expand it to f16 in the
// swizzled operand layout (exact for every int8 value); the MMA then runs in f16 with fp32
// accumulation, which is exact for integer partial sums below 2^24.  With WQ = 3 (full quant,
// decode orientation) the int8 activation tile comes with the weight tile and is expanded the
// same way, so the activation needs no kernel of its own and is read before the dependency.
//
// In the decode orientation a unit may hold MT = 2 row tiles of A (256 weight rows): one TMA box
// brings both, and two MMAs per K step share the B tile, so each weight byte costs half the
// activation traffic and half the TMA operations.
//
// With ALD the activation operand does not go through TMA: four loader warps copy it from global
// memory (where it sits in L2: it is small and was just written by the previous kernel) with
// 16-byte cp.async straight into the swizzled operand layout, and each loader thread's arrival
// on the stage's full barrier fires when its copies land.  TMA then carries only the weight
// stream, which is what a memory-bound decode GEMM needs: the activation tile per K step is as
// large as the weight tile, and sharing the TMA unit's requests with it halved the weight rate.
//
// With CG = 2 a cluster of two CTAs (a CTA pair on one TPC) computes each 256 x BN tile with
// tcgen05.mma.cta_group::2: each CTA stages its own 128 rows of A and half of the BN rows of B,
// the pair's first CTA issues the MMAs (M = 256), and each CTA's tensor memory receives the
// accumulator of its own 128 rows.  Per MMA FLOP a CTA then loads and holds a third less operand
// data, so 6 instead of 4 stages fit and more of the load latency is hidden (prefill).  Both
// CTAs' TMA loads complete on the first CTA's full barriers; its commits arrive on the stage and
// accumulator barriers of both CTAs; the second CTA's epilogue warps release an accumulator on
// the first CTA's barrier.
//
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer, warp 2 = TMEM owner, warp 3 = idle,
// warps 4..7 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31), warps 8..11 = int8 converters
// (WQ) or activation loaders (ALD).
//
// Work units: (m tile, n tile, batch, k split), m fastest, distributed round-robin over a grid
// of at most one CTA per SM.  Either operand may be "segmented": tiles below *_seg_tiles come
// from the first tensor map, the rest from the second (rebased to row 0), which lets one GEMM
// run over two separately stored weights (W^DQ and W^DKV|W^KR) without copying them together.
#pragma once
#include "ptx.cuh"
#include "stamps.cuh"

namespace mlap {

struct GemmGeometry {
  int32_t m_tiles, n_tiles, batches, splits;
  int32_t k_blocks;                 // ceil(K / 64)
  int32_t a_seg_tiles, b_seg_tiles; // tiles of A (B) served by the first map
  int32_t a_x_batch, a_y_batch;     // per-batch offsets of the TMA coordinates (elements, rows)
  int32_t b_x_batch, b_y_batch;
  int32_t num_units;
  int32_t w_op;                     // operand holding the weight: 0 = A, 1 = B
  // ALD: the activation operand (B, decode orientation) as a row-major bf16 matrix
  const uint16_t* act;              // element (y, x) at act[y * act_ld + x]
  int64_t act_ld;
  int32_t act_rows, act_cols;       // extents; copies outside them are zero-filled
  // Row-range schedule (weight as operand B, m_tiles = 1, no K split): the B rows of all batches,
  // batches * rr_rows in 32-row chunks, are cut into one equal contiguous range per CTA, and a
  // range into pieces at batch boundaries and every BN rows.  A piece is loaded as 32-row TMA
  // boxes and multiplied with N = its row count, so every SM streams the same share of the
  // weight whatever its row count (no tile rounding, no partial sums).
  int32_t rr_rows;
  // Optional execution stamps (%globaltimer) of this launch, kernel slot stamp_k (stamps.cuh).
  uint64_t* stamps;
  int32_t stamp_k;
  // 1: units walk the N tiles fastest (the A tiles are the large operand, e.g. the activations of
  // the prefill down-projection); 0: the M tiles fastest.
  int32_t n_fast;
  // 1: neither operand comes from an earlier kernel of the stream (both are inputs of the call),
  // so loads and MMAs start at once and only the epilogue waits for the preceding kernel, before
  // its first store (the preceding kernels may still read what it overwrites).
  int32_t act_ready;
};

// One piece of work for a CTA: a tile and its k-block range.
struct Frag {
  int tm, tn, b, s;
  int kb0, kb1;
  int row0, rows;   // row-range schedule: rows of operand B (within batch b) of the piece
};

// One TMA store of an epilogue staging tile: which output map, its rank and coordinates, and the
// tile's byte offset inside the warp's staging buffer.
struct StoreOp {
  int32_t which;   // 0: first output map, 1: second
  int32_t rank;    // 2 or 3
  int32_t x, y, z;
  uint32_t soff;
};

// WQ: 0 = bf16 weight, 1 = int8 weight in operand A, 2 = int8 weight in operand B, 3 = int8
//     weight in operand A and int8 activation in operand B (decode orientation, full quant: both
//     raw tiles arrive on the stage's raw barrier and the converter warps expand both).
// MT: 128-row tiles of A per unit (1 or 2), each with its own TMEM accumulator.
// ALD: operand B (the activation, decode orientation) is loaded by cp.async loader warps.
template <int BN_, int WQ_ = 0, int MT_ = 1, int ALD_ = 0, int CG_ = 1>
struct GemmCfg {
  static constexpr int CG = CG_;                       // CTAs per MMA (cta_group)
  static constexpr int WQ = WQ_;
  static constexpr int MT = MT_;
  static constexpr int ALD = ALD_;
  static constexpr int BM = 128;                       // rows per MMA
  static constexpr int BM_U = BM * MT;                 // rows of A per unit and CTA
  static constexpr int ROWS_U = BM_U * CG;             // rows of A per unit
  static constexpr int BN = BN_;
  static constexpr int BN_CTA = BN / CG;               // rows of B staged per CTA
  static constexpr int BK = 64;
  static constexpr int A_BYTES = BM_U * BK * 2;
  static constexpr int B_BYTES = BN_CTA * BK * 2;
  static constexpr int RAW_ROWS = (WQ == 1 || WQ == 3) ? BM_U : (WQ == 2 ? BN : 0);
  static constexpr int RAW_ACT_ROWS = WQ == 3 ? BN : 0;   // int8 activation rows (WQ = 3)
  static constexpr int RAW_W_BYTES = RAW_ROWS * BK;       // int8 weight tile
  static constexpr int RAW_BYTES = RAW_W_BYTES + RAW_ACT_ROWS * BK;   // a stage's int8 tiles
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + RAW_BYTES;
  static constexpr int SMEM_LIMIT = 232448;            // 227 KB opt-in per CTA
  static constexpr int RESERVED = 1024 + 512;          // alignment slack + barriers
  static constexpr int EPI_BUF = 4096;                 // one staging tile (32 x 32 fp32)
  static constexpr int EPI_BYTES = 4 * 2 * EPI_BUF;    // 4 epilogue warps, double-buffered
  static constexpr int STAGES_FIT = (SMEM_LIMIT - RESERVED - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + RESERVED;
  static constexpr int CH = BN >= 32 ? 32 : BN;        // epilogue column chunk
  static constexpr int ACC_COLS = 2 * MT * BN;         // double-buffered accumulators
  static constexpr uint32_t TMEM_COLS =
      ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64 : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
  // int8 weights run in f16 (the converters' output and the int8 paths' activations), else bf16
  static constexpr uint32_t IDESC = WQ ? idesc_f16_f32(BM * CG, BN) : idesc_bf16_f32(BM * CG, BN);
  static constexpr int THREADS = (WQ || ALD) ? 384 : 256;
  static constexpr uint32_t FULL_ARRIVALS = WQ ? 1 + 4 : (ALD ? 1 + 128 : 1);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N must be a multiple of 16 in [16,256]");
  static_assert(B_BYTES % 1024 == 0 && RAW_BYTES % 1024 == 0, "stages must keep 1024-B alignment");
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(ACC_COLS <= 512, "accumulators exceed tensor memory");
  static_assert(MT == 1 || MT == 2, "one or two row tiles per unit");
  static_assert(!(ALD && WQ), "cp.async activation loading is for bf16 weights");
  static_assert(CG == 1 || (CG == 2 && WQ == 0 && MT == 1 && ALD == 0 && BN % 32 == 0),
                "CTA-pair tiles: bf16 operands through TMA, one row tile, B split in halves");
};

__device__ __forceinline__ void decode_unit(const GemmGeometry& g, int u, int& tm, int& tn, int& b,
                                            int& s) {
  if (g.n_fast) {   // units of one A tile run together: the A tile is read from DRAM once
    tn = u % g.n_tiles;
    u /= g.n_tiles;
    tm = u % g.m_tiles;
    u /= g.m_tiles;
  } else {
    tm = u % g.m_tiles;
    u /= g.m_tiles;
    tn = u % g.n_tiles;
    u /= g.n_tiles;
  }
  b = u % g.batches;
  s = u / g.batches;
}

// Iterates this CTA's work; every role walks the same sequence.  RR: the row-range schedule
// (compile-time, so that the other launches carry none of its code).
template <bool RR, int BN>
struct FragIter {
  int u, step;
  long long i, i1;
  // first unit and stride: this CTA's index and the grid (one CTA per unit), or the pair's index
  // and the number of pairs (CTA pairs)
  __device__ __forceinline__ FragIter(const GemmGeometry& g, int first, int stride) {
    u = first;
    step = stride;
    i = i1 = 0;
    if constexpr (RR) {   // chunk range of this CTA
      const long long total = static_cast<long long>(g.batches) * (g.rr_rows / 32);
      i = total * blockIdx.x / gridDim.x;
      i1 = total * (blockIdx.x + 1) / gridDim.x;
    }
  }
  __device__ __forceinline__ bool next(const GemmGeometry& g, Frag& f) {
    if constexpr (RR) {
      if (i >= i1) return false;
      const int per_batch = g.rr_rows / 32;
      const int b = static_cast<int>(i / per_batch);
      const int c0 = static_cast<int>(i % per_batch);
      long long n = i1 - i;
      if (n > per_batch - c0) n = per_batch - c0;
      if (n > BN / 32) n = BN / 32;
      f.tm = 0;
      f.tn = 0;
      f.b = b;
      f.s = 0;
      f.kb0 = 0;
      f.kb1 = g.k_blocks;
      f.row0 = c0 * 32;
      f.rows = static_cast<int>(n) * 32;
      i += n;
      return true;
    }
    if (u >= g.num_units) return false;
    decode_unit(g, u, f.tm, f.tn, f.b, f.s);
    f.kb0 = (f.s * g.k_blocks) / g.splits;
    f.kb1 = ((f.s + 1) * g.k_blocks) / g.splits;
    f.row0 = 0;
    f.rows = 0;
    u += step;
    return true;
  }
};

// int8 to f16 by the 2^10 magic number: with u = v + 128 in [0, 255] (v XOR 0x80 per byte), the
// f16 with bits 0x6400 | u is 1024 + u exactly (f16 has 10 mantissa bits), so one byte permute
// builds two such halves and one packed f16 subtraction of 1024 + 128 gives v exactly.  The int8
// paths therefore run their MMAs with f16 operands (the c^Q codes and full quant's token_x are
// integers of magnitude <= 128 too, exact in f16): one permute and one packed subtract per two
// values, on the full-rate pipes.
__device__ __forceinline__ uint32_t int8x2_to_f16x2(uint32_t biased, uint32_t sel) {
  const uint32_t h = __byte_perm(biased, 0x64646464u, sel);
  __half2 v = *reinterpret_cast<const __half2*>(&h);
  v = __hsub2(v, __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6480u))));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// An int8 weight tile of `rows` 64-B rows to f16 in the 128B-swizzled K-major layout (row r,
// 16-byte chunk c at r*128 + ((c ^ (r & 7)) << 4)), by one thread of 128: the thread takes the
// source chunks ct, ct + 128, ... (row q / 4, chunk q % 4), so a warp's loads read 512 contiguous
// bytes and every thread has the same share of the tile.  All of a thread's loads are issued
// before any conversion (MAXC >= rows / 32 chunks per thread): the shared-memory latency is paid
// once per tile instead of once per chunk.
template <int MAXC>
__device__ __forceinline__ void convert_int8_tile(const uint8_t* raw, uint8_t* dst, int rows,
                                                  int ct) {
  const int n = rows * 4;
  uint4 v[MAXC];
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int q = ct + 128 * j;
    if (q < n) v[j] = *reinterpret_cast<const uint4*>(raw + q * 16);
  }
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int q = ct + 128 * j;
    if (q >= n) break;
    const int r = q >> 2, i = q & 3;
    const uint32_t w[4] = {v[j].x ^ 0x80808080u, v[j].y ^ 0x80808080u, v[j].z ^ 0x80808080u,
                           v[j].w ^ 0x80808080u};
    uint32_t out[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      out[2 * k] = int8x2_to_f16x2(w[k], 0x4140u);       // bytes 0, 1
      out[2 * k + 1] = int8x2_to_f16x2(w[k], 0x4342u);   // bytes 2, 3
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * i + h;
      *reinterpret_cast<uint4*>(dst + r * 128 + (((c ^ (r & 7)) & 7) << 4)) =
          make_uint4(out[4 * h], out[4 * h + 1], out[4 * h + 2], out[4 * h + 3]);
    }
  }
}

// Epilogue functor contract (see epilogues.cuh):
//   static constexpr int kCols;   // CH: the engine's chunk (32, or 16 when BN = 16), or 64
//   __device__ int operator()(int m0, int n0, int batch, int split, const float (&v)[kCols],
//                             uint8_t* stage, StoreOp (&ops)[2]) const;
// called by all 32 lanes of an epilogue warp together for the 32 x CH accumulator block whose
// first A row is m0 (lane l holds row m0 + l) and first B row is n0 (v[j] is column n0 + j).  It
// writes the block's output into the warp's staging buffer and returns the TMA stores (at most
// two, warp-uniform) that move it to global memory through the two output tensor maps.
template <int BN, class Epi, int WQ, int MT, int ALD, int CG>
__global__ void __launch_bounds__(GemmCfg<BN, WQ, MT, ALD, CG>::THREADS, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                     const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1,
                     const __grid_constant__ CUtensorMap tmO0,
                     const __grid_constant__ CUtensorMap tmO1, const GemmGeometry geo,
                     const Epi epi, uint32_t* __restrict__ err_word) {
  using Cfg = GemmCfg<BN, WQ, MT, ALD, CG>;
  constexpr bool RR = Epi::kDirect;   // the row-range launches are the direct-store ones
  static_assert(!(RR && CG == 2), "the row-range schedule runs on single CTAs");
  using Iter = FragIter<RR, BN>;
  // epilogue column chunk: the engine's 32 (16 for BN = 16) unless the functor asks for 64 (one
  // 128-byte bf16 row segment per lane and store)
  constexpr int ECH = Epi::kCols;
  static_assert(ECH == Cfg::CH || (ECH == 64 && Cfg::CH == 32 && BN % 64 == 0 && MT == 1),
                "epilogue chunk");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* smemA = smem;
  uint8_t* smemB = smemA + Cfg::STAGES * Cfg::A_BYTES;
  uint8_t* smemR = smemB + Cfg::STAGES * Cfg::B_BYTES;                  // raw int8 tiles
  uint8_t* smemE = smemR + Cfg::STAGES * Cfg::RAW_BYTES;                // epilogue staging
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smemE + Cfg::EPI_BYTES);
  uint64_t* empty_bar = full_bar + Cfg::STAGES;
  uint64_t* rawf_bar = empty_bar + Cfg::STAGES;
  uint64_t* accf_bar = rawf_bar + Cfg::STAGES;
  uint64_t* acce_bar = accf_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool w_is_a = geo.w_op == 0;
  // CTA pair: rank in the pair (0 issues the MMAs), the pair's units
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  const bool issuer = rank == 0;
  const int first_unit = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_step = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) stamp(geo.stamps, geo.stamp_k, kStampStart);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA0);
    prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB0);
    prefetch_tmap(&tmB1);
    prefetch_tmap(&tmO0);
    prefetch_tmap(&tmO1);
  }
  if (warp == 1 && lane == 0) {
    for (int i = 0; i < Cfg::STAGES; ++i) {
      mbar_init(&full_bar[i], Cfg::FULL_ARRIVALS);   // producer (+ converter warps / loader threads)
      mbar_init(&empty_bar[i], 1);
      mbar_init(&rawf_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf_bar[i], 1);
      mbar_init(&acce_bar[i], 4 * CG);   // the epilogue warps of every CTA of the pair
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 2) {
    if constexpr (CG == 2) {
      tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  if constexpr (CG == 2) cluster_sync();   // the peer's barriers exist before any remote arrival
  else __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // Let the next kernel in the stream start its prologue.  Every role except the producer waits
  // for the previous kernel's results here; the producer first requests weight tiles.
  grid_launch_dependents();
  const bool producer = warp == 0 && lane == 0;
  if (!producer && !geo.act_ready) grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      auto load_a = [&](int tm, int b, int kb, uint64_t* bar, void* dst) {
        const bool first = tm < geo.a_seg_tiles;
        const int y = (first ? tm : tm - geo.a_seg_tiles) * Cfg::ROWS_U +
                      static_cast<int>(rank) * Cfg::BM_U + b * geo.a_y_batch;
        const int x = kb * Cfg::BK + b * geo.a_x_batch;
        if constexpr (CG == 2)   // completes on the pair's first CTA's barrier
          tma_load_2d_pair(dst, first ? &tmA0 : &tmA1, mapa_shared(smem_u32(bar), 0), x, y);
        else
          tma_load_2d(dst, first ? &tmA0 : &tmA1, bar, x, y);
      };
      auto load_b = [&](const Frag& f, int kb, uint64_t* bar, void* dst) {
        const int tn = f.tn, b = f.b;
        if constexpr (RR) {   // 32-row boxes (single segment)
          for (int r = 0; r < f.rows; r += 32)
            tma_load_2d(static_cast<uint8_t*>(dst) + r * 128, &tmB0, bar,
                        kb * Cfg::BK + b * geo.b_x_batch, f.row0 + r + b * geo.b_y_batch);
          return;
        }
        const bool first = tn < geo.b_seg_tiles;
        const int y = (first ? tn : tn - geo.b_seg_tiles) * Cfg::BN +
                      static_cast<int>(rank) * Cfg::BN_CTA + b * geo.b_y_batch;
        const int x = kb * Cfg::BK + b * geo.b_x_batch;
        if constexpr (CG == 2)
          tma_load_2d_pair(dst, first ? &tmB0 : &tmB1, mapa_shared(smem_u32(bar), 0), x, y);
        else
          tma_load_2d(dst, first ? &tmB0 : &tmB1, bar, x, y);
      };
      // weight tile of stage st (bf16 into the operand buffer, or int8 into the raw buffer)
      auto issue_weight = [&](int st, const Frag& f, int kb) {
        if constexpr (WQ != 0) {
          mbar_arrive_expect_tx(&rawf_bar[st], Cfg::RAW_BYTES);
          if (WQ == 1 || WQ == 3) load_a(f.tm, f.b, kb, &rawf_bar[st], smemR + st * Cfg::RAW_BYTES);
          else load_b(f, kb, &rawf_bar[st], smemR + st * Cfg::RAW_BYTES);
          // the int8 activation tile rides with the weight's (an input of the call: no wait)
          if (WQ == 3)
            load_b(f, kb, &rawf_bar[st], smemR + st * Cfg::RAW_BYTES + Cfg::RAW_W_BYTES);
        } else if (ALD) {
          mbar_arrive_expect_tx(&full_bar[st], Cfg::A_BYTES);
          load_a(f.tm, f.b, kb, &full_bar[st], smemA + st * Cfg::A_BYTES);
        } else if (w_is_a) {
          // (a pair's stage completes on its first CTA's barrier: it expects both CTAs' bytes)
          if (issuer) mbar_expect_tx(&full_bar[st], CG * Cfg::A_BYTES);
          load_a(f.tm, f.b, kb, &full_bar[st], smemA + st * Cfg::A_BYTES);
        } else {
          if (issuer)
            mbar_expect_tx(&full_bar[st], RR ? static_cast<uint32_t>(f.rows) * Cfg::BK * 2
                                             : static_cast<uint32_t>(CG * Cfg::B_BYTES));
          load_b(f, kb, &full_bar[st], smemB + st * Cfg::B_BYTES);
        }
      };
      auto issue_act = [&](int st, const Frag& f, int kb) {
        if (ALD) return;
        if (WQ == 3) {   // the activation came with the weight's raw tiles: only the arrival
          mbar_arrive(&full_bar[st]);
          return;
        }
        if (w_is_a) {
          if (issuer) mbar_arrive_expect_tx(&full_bar[st], CG * Cfg::B_BYTES);
          load_b(f, kb, &full_bar[st], smemB + st * Cfg::B_BYTES);
        } else {
          if (issuer) mbar_arrive_expect_tx(&full_bar[st], CG * Cfg::A_BYTES);
          load_a(f.tm, f.b, kb, &full_bar[st], smemA + st * Cfg::A_BYTES);
        }
      };

      // Weight tiles of this CTA's first stages, before the grid dependency resolves.
      int pre = 0;
      {
        Iter it0(geo, first_unit, unit_step);
        Frag f0;
        if (it0.next(geo, f0)) {
          pre = f0.kb1 - f0.kb0 < Cfg::STAGES ? f0.kb1 - f0.kb0 : Cfg::STAGES;
          for (int i = 0; i < pre; ++i) issue_weight(i, f0, f0.kb0 + i);
        }
      }
      if (!geo.act_ready) {
        grid_dependency_wait();
        stamp(geo.stamps, geo.stamp_k, kStampDep);
      }

      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Iter it(geo, first_unit, unit_step);
      Frag f;
      for (int n = 0; ok && it.next(geo, f); ++n) {
        const int kb0 = f.kb0, kb1 = f.kb1;
        for (int kb = kb0; kb < kb1; ++kb) {
          const bool prefetched = n == 0 && kb - kb0 < pre;
          if (!prefetched) {
            // (a pair's stages are freed by the first CTA's MMA commits)
            const bool empty = CG == 2 ? mbar_wait_cluster(&empty_bar[stage], phase ^ 1u, abort_flag)
                                       : mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag);
            if (!empty) {
              ok = false;
              break;
            }
            issue_weight(stage, f, kb);
          }
          issue_act(stage, f, kb);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag && issuer) {
        // Give up cleanly: let every load already issued land before the CTA exits.  The last
        // fill of stage i has parity `phase` if i < stage (this lap), else `phase ^ 1`.  (A
        // pair's second CTA waits at the end instead: its loads complete on these barriers.)
        for (int i = 0; i < Cfg::STAGES; ++i) {
          const uint32_t par = (i < stage) ? phase : (phase ^ 1u);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full_bar[i], par) && globaltimer_ns() - t0 < 20000000ull) {
          }
          if (WQ) {
            while (!mbar_try_wait(&rawf_bar[i], par) && globaltimer_ns() - t0 < 20000000ull) {
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && issuer) {
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0;
      bool ok = true;
      Iter it(geo, first_unit, unit_step);
      Frag f;
      for (; ok && it.next(geo, f); ++iter) {
        const int kb0 = f.kb0, kb1 = f.kb1;
        const int buf = iter & 1;
        const uint32_t use = static_cast<uint32_t>(iter >> 1);
        const bool freed = CG == 2 ? mbar_wait_cluster(&acce_bar[buf], (use & 1u) ^ 1u, abort_flag)
                                   : mbar_wait(&acce_bar[buf], (use & 1u) ^ 1u, abort_flag);
        if (!freed) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * MT * Cfg::BN);
        const uint32_t idesc = RR ? idesc_bf16_f32(Cfg::BM, f.rows) : Cfg::IDESC;
        for (int kb = kb0; kb < kb1; ++kb) {
          const bool landed = CG == 2 ? mbar_wait_cluster(&full_bar[stage], phase, abort_flag)
                                      : mbar_wait(&full_bar[stage], phase, abort_flag);
          if (!landed) {
            ok = false;
            break;
          }
          if (ALD) fence_proxy_async_shared();   // cp.async (generic proxy) data -> tensor core
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(smemA + stage * Cfg::A_BYTES);
          const uint32_t b_addr = smem_u32(smemB + stage * Cfg::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < Cfg::BK / 16; ++kk) {
            if constexpr (CG == 2) {
              umma_bf16_ss_pair(d_tmem, sdesc_kmajor_sw128(a_addr + kk * 32),
                                sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                                (kb > kb0 || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
              for (int h = 0; h < MT; ++h)
                umma_bf16_ss(d_tmem + h * Cfg::BN,
                             sdesc_kmajor_sw128(a_addr + h * Cfg::BM * Cfg::BK * 2 + kk * 32),
                             sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                             (kb > kb0 || kk > 0) ? 1u : 0u);
            }
          }
          // frees this smem stage (in both CTAs of a pair) once the MMAs have read it
          if constexpr (CG == 2) umma_commit_pair(&empty_bar[stage], 0x3);
          else umma_commit(&empty_bar[stage]);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) {   // accumulator ready for the epilogue (of both CTAs of a pair)
          if constexpr (CG == 2) umma_commit_pair(&accf_bar[buf], 0x3);
          else umma_commit(&accf_bar[buf]);
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint8_t* wstage = smemE + q * 2 * Cfg::EPI_BUF;
    if (geo.act_ready) {   // the stores wait for the preceding kernel
      grid_dependency_wait();
      if (q == 0 && lane == 0) stamp(geo.stamps, geo.stamp_k, kStampDep);
    }
    int sel = 0;
    int iter = 0;
    Iter it(geo, first_unit, unit_step);
    Frag f;
    for (; it.next(geo, f); ++iter) {
      const int tm = f.tm, tn = f.tn, b = f.b, s = f.s;
      const int buf = iter & 1;
      const uint32_t use = static_cast<uint32_t>(iter >> 1);
      const int n_row0 = RR ? f.row0 : tn * Cfg::BN;            // this piece's B rows
      const int ncols = RR ? MT * f.rows : MT * Cfg::BN;        // accumulator columns
      // inputs the epilogue of the first block needs (e.g. RoPE tables), before the wait
      const int m_base = tm * Cfg::ROWS_U + static_cast<int>(rank) * Cfg::BM_U;   // this CTA's rows
      typename Epi::Pre pre = epi.preload(m_base + q * 32, n_row0);
      const bool ready = CG == 2 ? mbar_wait_cluster(&accf_bar[buf], use & 1u, abort_flag)
                                 : mbar_wait(&accf_bar[buf], use & 1u, abort_flag);
      if (!ready) break;
      tc_fence_after_sync();
      if (q == 0 && lane == 0) stamp(geo.stamps, geo.stamp_k, kStampMain);
#pragma unroll 1
      for (int hc = 0; hc < ncols; hc += ECH) {
        const int h = hc / Cfg::BN, c = hc % Cfg::BN;
        const int m0 = m_base + h * Cfg::BM + q * 32;
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(buf * MT * Cfg::BN + hc);
        float v[ECH];
        if constexpr (ECH == 64) {
          uint32_t r[32], r2[32];
          tmem_ld_32x32b_x32(t_addr, r);
          tmem_ld_32x32b_x32(t_addr + 32, r2);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = __uint_as_float(r[j]);
            v[32 + j] = __uint_as_float(r2[j]);
          }
        } else if constexpr (ECH == 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_addr, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        } else {
          uint32_t r[16];
          tmem_ld_32x32b_x16(t_addr, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
        }
        if (hc + ECH >= ncols) {
          // last TMEM read of this accumulator: hand it back to the MMA warp right away
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {   // (a pair's accumulators are released on its first CTA's barrier)
            if constexpr (CG == 2) mbar_arrive_cluster(mapa_shared(smem_u32(&acce_bar[buf]), 0));
            else mbar_arrive(&acce_bar[buf]);
          }
        }
        uint8_t* sb = wstage + sel * Cfg::EPI_BUF;
        sel ^= 1;
        if (lane == 0) bulk_wait_group_read<1>();   // the store that last read this buffer is done
        __syncwarp();
        StoreOp ops[2];
        const int nops = epi(m0, n_row0 + c, b, s, v, sb, ops, pre);
        if (hc + ECH < ncols) {   // the next block's inputs, while this one stores
          const int hn = (hc + ECH) / Cfg::BN, cn = (hc + ECH) % Cfg::BN;
          pre = epi.preload(m_base + hn * Cfg::BM + q * 32, n_row0 + cn);
        }
        if constexpr (Epi::kDirect) continue;   // written directly from registers
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          for (int i = 0; i < nops; ++i) {
            const CUtensorMap* m = ops[i].which ? &tmO1 : &tmO0;
            if (ops[i].rank == 2)
              tma_store_2d(m, sb + ops[i].soff, ops[i].x, ops[i].y);
            else
              tma_store_3d(m, sb + ops[i].soff, ops[i].x, ops[i].y, ops[i].z);
          }
          bulk_commit_group();
        }
      }
    }
    // every store has read its staging buffer (the writes themselves complete with the grid)
    if (lane == 0) bulk_wait_group_read<0>();
  } else if (WQ != 0 && warp >= 8) {
    // ------------------------------------------------------------------ int8 -> f16 converters
    const int ct = threadIdx.x - 256;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    Iter it(geo, first_unit, unit_step);
    Frag f;
    while (ok && it.next(geo, f)) {
      for (int kb = f.kb0; kb < f.kb1; ++kb) {
        if (!mbar_wait(&rawf_bar[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smemR + stage * Cfg::RAW_BYTES;
        uint8_t* dst = (WQ == 1 || WQ == 3) ? smemA + stage * Cfg::A_BYTES
                                            : smemB + stage * Cfg::B_BYTES;
        constexpr int kChunks = Cfg::RAW_ROWS ? (Cfg::RAW_ROWS + 31) / 32 : 1;   // per thread
        convert_int8_tile<kChunks>(raw, dst, Cfg::RAW_ROWS, ct);
        if constexpr (WQ == 3) {   // the int8 activation tile into operand B
          constexpr int kActChunks = (Cfg::RAW_ACT_ROWS + 31) / 32;
          convert_int8_tile<kActChunks>(raw + Cfg::RAW_W_BYTES, smemB + stage * Cfg::B_BYTES,
                                        Cfg::RAW_ACT_ROWS, ct);
        }
        fence_proxy_async_shared();              // generic writes -> visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_bar[stage]);
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (ALD && warp >= 8) {
    // ------------------------------------------------------------------ activation loaders
    // Thread t copies 16-byte chunk (t % 8) of rows t / 8, t / 8 + 16, ... of the BN x 64 tile:
    // eight consecutive lanes read one 128-byte row segment.
    const int lt = threadIdx.x - 256;
    const int c = lt & 7;
    const int r0 = lt >> 3;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    Iter it(geo, first_unit, unit_step);
    Frag f;
    while (ok && it.next(geo, f)) {
      const int y0 = f.tn * Cfg::BN + f.b * geo.b_y_batch;
      for (int kb = f.kb0; kb < f.kb1; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const int x = f.b * geo.b_x_batch + kb * Cfg::BK + c * 8;
        const bool xin = x < geo.act_cols;
        uint8_t* dst = smemB + stage * Cfg::B_BYTES;
#pragma unroll
        for (int i = 0; i < Cfg::BN / 16; ++i) {
          const int r = r0 + 16 * i;
          const int y = y0 + r;
          const bool in = xin && y < geo.act_rows;
          const uint16_t* src = in ? geo.act + static_cast<int64_t>(y) * geo.act_ld + x : geo.act;
          cp_async_16(dst + r * 128 + (((c ^ (r & 7)) & 7) << 4), src, in ? 16u : 0u);
        }
        cp_async_arrive_noinc(&full_bar[stage]);
        if (++stage == Cfg::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    cp_async_wait_all();                         // nothing of ours lands after the CTA exits
  }

  __syncthreads();
  if constexpr (CG == 2) {
    // After a timeout this CTA may still have loads in flight that complete on the other CTA's
    // barriers: give them time to land (bounded) before the shared memory goes away.
    if (*abort_flag) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) {
      }
    }
    // both CTAs' epilogues have read their accumulators before the pair frees tensor memory
    tc_fence_before_sync();
    cluster_sync();
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(err_word, kErrTimeout);
  if (threadIdx.x == 0) stamp(geo.stamps, geo.stamp_k, kStampEnd);
  if (warp == 2) {
    tc_fence_after_sync();
    if constexpr (CG == 2) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace mlap
