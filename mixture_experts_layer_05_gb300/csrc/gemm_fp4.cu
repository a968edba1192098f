// NVFP4 (w4a4, 16-value blocks with e4m3 scales and a per-tensor fp32 scale) grouped GEMMs
// of the FusedMoE expert MLP, the FlashInferFP4MoE layer of the sglang
// `fused_moe_triton/layer.py` page (`trtllm_fp4_block_scale_moe` with `gemm1_weights` /
// `gemm2_weights` and their block scales):
//
//   w13: z[f][n] = alpha_e * sum_k xq[row][k] w13q[e][n][k]   fp32 partials, n in [0, 2I)
//   w2 : o = alpha_e * sum_k aq[row][k] w2q[e][n][k], times the routing weight, to the
//        token's fp32 slot
//
// with xq / aq the f16 values q * sf of the quantized rows (exact) and w q * sf of the
// weights (exact in f16), alpha_e = weight_scale_2[e] / g (g the rows' per-tensor scale).
//
// The weights arrive prepared (moe_nvfp4_prepare_weight): per tile of 128 rows and K stage
// of 64 values one contiguous 4608-byte chunk, the packed codes of the stage's two K halves
// (16 bytes per row each) then the rows' four scale bytes. A unit is a row block of up to
// 128 token rows against 256 weight rows (128 when the weight rows do not split into 256s)
// over a K range of whole 128-value stages.
//
// The tensor core's time per MMA follows N, not M (M 128 x K 16 costs about 45 cycles at
// N = 16 or 32, 48 at 64, 64 at 128 and 128 at N = 256, the same for M = 64), so the unit's
// tokens go on N and the expanded weights are the A operand (M 128 per weight tile), written
// by the converters straight into tensor memory (tcgen05.st): no f16 weight tile
// round-trips through shared memory, which carries only the chunk copies and the token
// tiles. Roles:
//
//   warp 0       bulk copies (one 9216-byte piece per weight tile and stage: the tile's two
//                chunks are consecutive along K) into an 8-deep raw ring
//   warp 2       the stage's two token boxes (16 / 32 / 64 / 128 rows x 64 values) into slot
//                (stage mod S) of the token ring, completing on that stage's barrier (S =
//                the TMEM A ring's stages)
//   warp 3       the unit scheduler: reads each unit's metadata from global memory ahead
//                of time and publishes it in shared memory
//   warps 1,     four MMA issuers: M 128 (weights, A in TMEM) x N (the unit's token rows
//   24..26       rounded to 16) x K 16, one stage barrier wait and one commit per stage
//                each; issuer q takes weight tile q / 2 and the stage's K chunk q % 2 (4
//                MMAs per stage into its own accumulator), or, for 128-row token boxes,
//                issuers 0 and 1 take tile q (8 MMAs per stage). A thread's tcgen05.mma
//                issue, not the tensor core, bounds this kernel's MMA side: one issuer for
//                both tiles was 30 % slower than two, four are 10-15 % faster than two.
//   warps 4..19  two groups of 8 on alternate stages: warp c expands weight row
//                32 (c % 4) + lane of tile (c / 4) % 2, both K chunks of the stage (codes
//                and block scales, one hardware e2m1x2 conversion and one packed multiply
//                per pair) into 64 TMEM columns of the stage's A slot (its lane quarter)
//   warps 20..23 epilogue: TMEM lane = output column, TMEM column = token row
//
// TMEM holds the accumulators (four or two per buffer; two buffers, alternate units, for
// 16-row boxes, else one, so a unit's MMAs wait for the previous unit's epilogue), then the
// A ring. (Releasing a buffer's two tiles one at a time, each to its own issuer, measured
// 1-3 % slower.) Every wait is bounded (kWaitTimeoutNs).
#include "fp4.cuh"
#include "tc.cuh"

namespace gbmoe {
namespace {

constexpr int kF4TileRows = 128;                  // rows of a prepared tile
constexpr int kF4MaxN = 256;                      // weight rows per unit
constexpr int kF4M = 128;                         // weight rows per MMA (M)
constexpr int kF4BK = kFp4StageK;                 // K values per prepared chunk and token box
constexpr int kF4StageK = 2 * kFp4StageK;         // K values per stage
constexpr uint32_t kF4Piece = 2 * kFp4ChunkBytes; // a tile's chunks of one stage
constexpr uint32_t kF4RawBytes = 2 * kF4Piece;    // two tiles
constexpr int kF4RawStages = 8;
constexpr int kF4MaxRows = 128;                   // token rows per unit (MMA N)
constexpr int kF4MaxSlots = 4;                    // weight stages in TMEM (and token slots)
constexpr uint32_t kF4TokArea = 64 * 1024;        // token ring: up to 2 stages of 2 x 16 KB
constexpr int kF4CvtWarps = 16;
constexpr int kF4EpiWarps = 4;
constexpr int kF4Issuers = 4;                     // MMA-issuing warps: 1 and 24..26
constexpr int kF4Threads = 32 * (3 + kF4Issuers + kF4CvtWarps + kF4EpiWarps);
constexpr int kF4Issuer1 = 4 + kF4CvtWarps + kF4EpiWarps;         // warp of issuer 1 (24)
constexpr uint32_t kF4TmemCols = 512;
constexpr int kF4Boxes = 4;                       // token boxes of 16, 32, 64, 128 rows
constexpr int kF4UnitRing = 8;                    // unit descriptors the scheduler runs ahead
// arrivals that free a descriptor: the two producers, the MMA issuers, every converter warp
// and every epilogue warp
constexpr int kF4UnitReaders = 2 + kF4Issuers + kF4CvtWarps + kF4EpiWarps;
constexpr uint32_t kF4BarBytes = 2048;
constexpr size_t kF4Smem = 1024 + kF4TokArea + (size_t)kF4RawStages * kF4RawBytes + kF4BarBytes;
static_assert(kF4Smem <= 232448, "shared memory per CTA exceeded");
static_assert(kF4Piece % 16 == 0, "bulk copies move multiples of 16 bytes");
// TMEM: the accumulators, then the A ring, 128 columns (two tiles x 128 f16 values) per
// stage. Four accumulators per buffer, one per MMA-issuing warp, acc columns each (the
// launch's widest token box, at most 64): for a unit of at most 64 token rows accumulator q
// holds weight tile q / 2 and the stage's K chunk q % 2 (the epilogue adds a tile's two in
// a fixed order); for a wider unit accumulators 2 t and 2 t + 1 hold tile t's token rows
// 0..63 and 64..127, one 128-column accumulator. Two buffers (alternate units) when three A
// stages still fit, else one.
__host__ __device__ constexpr int f4_acc(int box_rows) { return box_rows < 64 ? box_rows : 64; }
__host__ __device__ constexpr int f4_bufs(int box_rows) {
  return 2 * 4 * f4_acc(box_rows) + 3 * 128 <= (int)kF4TmemCols ? 2 : 1;
}
__host__ __device__ constexpr int f4_acc_cols(int box_rows) {
  return f4_bufs(box_rows) * 4 * f4_acc(box_rows);
}
__host__ __device__ constexpr int f4_slots(int box_rows) {
  return ((int)kF4TmemCols - f4_acc_cols(box_rows)) / 128 < kF4MaxSlots
             ? ((int)kF4TmemCols - f4_acc_cols(box_rows)) / 128
             : kF4MaxSlots;
}
static_assert(f4_slots(16) == 3 && f4_slots(32) == 3 && f4_slots(64) == 2 &&
                  f4_slots(kF4MaxRows) == 2 &&
                  f4_slots(16) * 2 * 16 * 128 <= (int)kF4TokArea &&
                  f4_slots(32) * 2 * 32 * 128 <= (int)kF4TokArea &&
                  f4_slots(64) * 2 * 64 * 128 <= (int)kF4TokArea &&
                  f4_slots(kF4MaxRows) * 2 * kF4MaxRows * 128 <= (int)kF4TokArea,
              "rings");

struct F4Maps {
  CUtensorMap x[2][kF4Boxes];  // per problem: f16 token rows, box 64 values x (16 << i) rows
  int slots;                   // stages of the TMEM A ring and of the token ring
  int tok_slot_bytes;          // two boxes of the launch's widest box (a multiple of 2048)
  int box_rows;                // the launch's widest token box (16, 32, 64 or 128 rows)
  int un;                      // weight rows per unit: 256, or 128
  int acc_stride;              // TMEM columns per accumulator (box rows, at most 64)
};

// Instruction descriptor of kind::f16 with f16 A and B (format code 0), fp32 D, K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// The two e4m3 block scales of a 16-bit word (low byte first) as f16 pairs {s, s} (exact).
__device__ __forceinline__ void e4m3x2_pairs(uint32_t w, uint32_t& s0, uint32_t& s1) {
  asm("{\n\t.reg .b16 lo, hi;\n\t.reg .b32 p;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 p, lo;\n\t"
      "prmt.b32 %0, p, 0, 0x1010;\n\t"
      "prmt.b32 %1, p, 0, 0x3232;\n\t}"
      : "=r"(s0), "=r"(s1)
      : "r"(w));
}

// The eight e2m1 values of a word (element 2i in the low nibble of byte i) as four f16
// pairs, each multiplied by the f16 pair sc (exact: both factors have few significant bits).
__device__ __forceinline__ void e2m1x8_scaled(uint32_t w, uint32_t sc, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 h0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
      "mul.rn.f16x2 %0, h0, %5;\n\t"
      "mul.rn.f16x2 %1, h1, %5;\n\t"
      "mul.rn.f16x2 %2, h2, %5;\n\t"
      "mul.rn.f16x2 %3, h3, %5;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w), "r"(sc));
}

// 32 lanes x 32 consecutive 32-bit TMEM columns from registers (this warp's lane quarter).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
      "%27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, f16 inputs (A: lane = row, column c = values 2c, 2c + 1).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Spin (bounded, ignoring the abort flag) until the phase of `bar` with parity `parity`
// has completed: the producers' last copies must land before the CTA exits.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > 10000000ull) return;
}

// wait_bounded for a thread that only keeps pace (an idle MMA issuer): it sleeps between
// polls so that its spinning does not take issue slots from the warps doing the work.
__device__ __noinline__ bool wait_sleepy(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(256);
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      record_status(status, GBMOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// A unit as the scheduler warp publishes it in shared memory: the unit, its real token
// rows, its MMA N (rows rounded up to 16) and token box, its expert's first weight tile, the
// output scale.
struct F4Desc {
  int p, split, mb, nt, kb0, kb1, rows, n, box, tile;
  float alpha;
  int pad;
};
static_assert(sizeof(F4Desc) == 48, "descriptor size");

// Unit u: the row block's real rows (the align's per-block counts bounded by the launch's
// rows_bound, for routed problems; the identity rows left, for the shared one), that count
// rounded up to 16 and the smallest token box that holds them.
__device__ __forceinline__ F4Desc f4_desc(const GemmLaunch& L, const Schedule& S, int u, int un) {
  const Unit w = S.unit(L, u);
  const GemmProblem& P = L.p[w.p];
  int rows;
  if (P.sorted_ids)
    rows = P.block_rows ? min(P.block_rows[w.mb], P.rows_bound) : P.rows_bound;
  else
    rows = P.store_rows - w.mb * kFp4BS;
  rows = rows < 1 ? 1 : (rows > kFp4BS ? kFp4BS : rows);
  int e = P.expert_ids ? P.expert_ids[w.mb] : 0;
  if ((unsigned)e >= (unsigned)P.num_experts) {
    record_status(L.status, GBMOE_ERR_DEVICE_CHECK);
    e = 0;
  }
  F4Desc d;
  d.p = w.p;
  d.split = w.split;
  d.mb = w.mb;
  d.nt = w.nt;
  d.kb0 = w.kb0;
  d.kb1 = w.kb1;
  d.rows = rows;
  d.n = (rows + 15) & ~15;
  d.box = d.n <= 16 ? 0 : (d.n <= 32 ? 1 : (d.n <= 64 ? 2 : 3));
  d.tile = (int)(((long long)e * P.b_rows_per_expert + (long long)w.nt * un) / kF4TileRows);
  d.alpha = __fdiv_rn(P.scale2 ? P.scale2[e] : 1.f, P.gscale);
  d.pad = 0;
  return d;
}

// A ring position: slot and phase parity, advanced without division.
struct RingPos {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

template <int KIND>
__global__ void __launch_bounds__(kF4Threads, 1)
    gemm_fp4_kernel(const __grid_constant__ F4Maps maps, const __grid_constant__ GemmLaunch args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw0 = smem_addr(smem_raw);
  const uint32_t base = (raw0 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw0);
  // [token ring 64 KB] [raw ring 8 x 18 KB] [barriers, TMEM slot, abort flag, descriptors]
  const int nslots = maps.slots;
  const uint32_t acc_stride = (uint32_t)maps.acc_stride;
  const uint32_t box_rows = (uint32_t)maps.box_rows;
  const int nbuf = f4_bufs(maps.box_rows);                    // accumulator buffers
  const uint32_t a_col = (uint32_t)f4_acc_cols(maps.box_rows);  // first A ring column
  const uint32_t tsb = (uint32_t)maps.tok_slot_bytes;
  const int un = maps.un;
  const int chunks = un / kF4TileRows;             // weight tiles per unit: 1 or 2
  const uint32_t tok_base = base;
  const uint32_t raw_base = tok_base + kF4TokArea;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF4TokArea + kF4RawStages * kF4RawBytes);
  // bars: raw_full[8] raw_empty[8] stage_full[4] stage_empty[4] tfull[2] tempty[2]
  //       unit_full[8] unit_empty[8]; then the TMEM slot, the abort flag and (at byte 1024)
  //       the unit descriptors
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 44);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  F4Desc* descs = reinterpret_cast<F4Desc*>(reinterpret_cast<uint8_t*>(bars) + 1024);
  const uint32_t bar0 = smem_addr(bars);
  auto raw_full = [&](int s) { return bar0 + 8u * s; };
  auto raw_empty = [&](int s) { return bar0 + 8u * (8 + s); };
  auto stage_full = [&](int s) { return bar0 + 8u * (16 + s); };
  auto stage_empty = [&](int s) { return bar0 + 8u * (20 + s); };
  auto tfull = [&](int b) { return bar0 + 8u * (24 + b); };
  auto tempty = [&](int b) { return bar0 + 8u * (26 + b); };
  auto unit_full = [&](int i) { return bar0 + 8u * (28 + i); };
  auto unit_empty = [&](int i) { return bar0 + 8u * (36 + i); };
  auto x_stage = [&](int s) { return tok_base + s * tsb; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4RawStages; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(raw_empty(s), kF4CvtWarps / 2);   // the stage's converter group
    }
    for (int s = 0; s < nslots; ++s) {
      mbar_init(stage_full(s), kF4CvtWarps / 2 + 1);  // its converter group + token expect_tx
      mbar_init(stage_empty(s), 2 * chunks);      // one commit per active issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 2 * chunks);
      mbar_init(tempty(b), kF4EpiWarps);
    }
    for (int i = 0; i < kF4UnitRing; ++i) {
      mbar_init(unit_full(i), 1);
      mbar_init(unit_empty(i), kF4UnitReaders);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2 && lane == 0) {
    for (int p = 0; p < args.num_problems; ++p)
      for (int i = 0; i < kF4Boxes; ++i) tma_prefetch(&maps.x[p][i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kF4TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the token rows and the routing are earlier kernels' outputs
  if (threadIdx.x == 0) pdl_trigger();

  Schedule sched;
  sched.init(args, kFp4BS);
  // the next unit of this CTA from the scheduler warp's ring, as a copy in registers; every
  // reading warp releases the slot once
  auto get_unit = [&](const RingPos& q, F4Desc& d) -> bool {
    if (!wait_fast(unit_full(q.slot), q.phase, abort_flag, args.status)) return false;
    d = descs[q.slot];
    return true;
  };
  auto release_unit = [&](RingPos& q) {
    __syncwarp();
    if (lane == 0) mbar_arrive(unit_empty(q.slot));
    q.next(kF4UnitRing);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ prepared weight chunks
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      RingPos uq{0, 0}, rq{0, 0};
      uint32_t issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
        F4Desc w;
        if (!get_unit(uq, w)) break;
        mbar_arrive(unit_empty(uq.slot));
        uq.next(kF4UnitRing);
        const GemmProblem& P = args.p[w.p];
        const uint8_t* src = static_cast<const uint8_t*>(P.B) +
                             ((size_t)w.tile * P.k_blocks + w.kb0) * (size_t)kF4Piece;
        const size_t tile_bytes = (size_t)P.k_blocks * kF4Piece;  // the next tile's chunks
        for (int kb = w.kb0; kb < w.kb1;
             ++kb, src += kF4Piece, rq.next(kF4RawStages), ++issued) {
          if (!wait_fast(raw_empty(rq.slot), rq.phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(raw_full(rq.slot), chunks * kF4Piece);
          const uint32_t dst = raw_base + rq.slot * kF4RawBytes;
          for (int c = 0; c < chunks; ++c)
            bulk_load(dst + c * kF4Piece, src + c * tile_bytes, kF4Piece, raw_full(rq.slot),
                      policy);
        }
      }
      // the last copies of each slot land before the CTA can exit
      for (uint32_t j = issued > (uint32_t)kF4RawStages ? issued - kF4RawStages : 0; j < issued;
           ++j)
        drain_wait(raw_full(j % kF4RawStages), (j / kF4RawStages) & 1u);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ token tiles
    // The token tile of stage j lands in slot j of the token ring (two boxes of 64 values,
    // the second box_rows rows after the first) and completes on that stage's barrier, so
    // the MMA issuers wait once per stage.
    if (lane == 0) {
      RingPos uq{0, 0}, tq{0, 0};
      uint32_t issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
        F4Desc w;
        if (!get_unit(uq, w)) break;
        mbar_arrive(unit_empty(uq.slot));
        uq.next(kF4UnitRing);
        const CUtensorMap* map = &maps.x[w.p][w.box];
        const uint32_t box_bytes = (uint32_t)(16 << w.box) * 128;
        for (int kb = w.kb0; kb < w.kb1; ++kb, tq.next(nslots), ++issued) {
          if (!wait_fast(stage_empty(tq.slot), tq.phase ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(stage_full(tq.slot), 2 * box_bytes);
          tma_load_2d(x_stage(tq.slot), map, stage_full(tq.slot), kb * kF4StageK,
                      w.mb * kFp4BS);
          tma_load_2d(x_stage(tq.slot) + box_rows * 128u, map, stage_full(tq.slot),
                      kb * kF4StageK + kF4BK, w.mb * kFp4BS);
        }
      }
      const uint32_t n = (uint32_t)nslots;
      for (uint32_t j = issued > n ? issued - n : 0; j < issued; ++j)
        drain_wait(stage_full(j % n), (j / n) & 1u);
    }
    __syncwarp();
  } else if (warp == 1 || (warp >= kF4Issuer1 && warp < kF4Issuer1 + kF4Issuers - 1)) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer q (warps 1, 25, 24, 26 for q = 0..3) takes weight tile q / 2. A unit of at
    // most 64 token rows: the stage's K chunk q % 2, 4 MMAs per stage into its own
    // accumulator q (the epilogue adds a tile's two). A wider unit: issuer 2 t takes all of
    // tile t, 8 MMAs of N = the unit's rows per stage into accumulators 2 t and 2 t + 1 side
    // by side (128 columns); its partner issues no MMAs but keeps the same protocol (every
    // wait, one arrival per stage and per unit), so every stage barrier gets its arrivals
    // from the same issuers in every unit and no issuer runs ahead of the stage ring. (A
    // partner that skipped the unit's stages instead could see a stage barrier two phases
    // on as complete, by parity, and over-arrive on it: that faulted the GPU.) One thread
    // issues into each accumulator, so its summation order is fixed. Issuers 0 and 2, a
    // wide unit's two, sit on different SM sub-partitions (warps 1 and 24).
    const int q = warp == 1 ? 0 : warp == kF4Issuer1 ? 2 : warp == kF4Issuer1 + 1 ? 1 : 3;
    const int mt = q >> 1, sub = q & 1;   // weight tile; K chunk
    if (lane == 0) {
      RingPos uq{0, 0}, cq{0, 0};
      uint32_t uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x, ++uc) {
        F4Desc w;
        if (!get_unit(uq, w)) break;
        mbar_arrive(unit_empty(uq.slot));
        uq.next(kF4UnitRing);
        if (mt >= chunks) continue;  // no second tile: this issuer only follows the units
        const bool wide = w.n > 64;
        const bool idle = wide && sub == 1;   // the partner issues this unit's MMAs
        // weights on M (128 rows per tile, A in TMEM), the unit's tokens on N; with one
        // accumulator buffer every unit waits for the previous unit's epilogue
        const uint32_t idesc = idesc_f16(kF4M, w.n);
        const int tb = nbuf == 2 ? (int)(uc & 1u) : 0;
        const uint32_t tph = nbuf == 2 ? ((uc >> 1) & 1u) : (uc & 1u);
        if (!wait_fast(tempty(tb), tph ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + ((uint32_t)tb * 4u + (uint32_t)q) * acc_stride;
        // K step kk: 32 bytes into the token rows' swizzled 128-byte atoms, 8 columns into
        // the weights' TMEM stage; the stage's second 64 K values sit in the token slot's
        // second box and in the tile's columns 32..63
        if (!wide) {
          const uint32_t boff = (uint32_t)sub * box_rows * 128u, aoff = (uint32_t)sub * 32u;
          for (int kb = w.kb0; kb < w.kb1; ++kb, cq.next(nslots)) {
            // the stage barrier: the weights in TMEM and the token tile in its slot
            if (!wait_fast(stage_full(cq.slot), cq.phase, abort_flag, args.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bk = sdesc_advance(sdesc_sw128(x_stage(cq.slot)), boff);
            const uint32_t ak = tmem_base + a_col + (uint32_t)cq.slot * 128u + mt * 64u + aoff;
            mma_f16_ts(d, ak, bk, idesc, kb == w.kb0 ? 0u : 1u);
            mma_f16_ts(d, ak + 8, sdesc_advance(bk, 32), idesc, 1u);
            mma_f16_ts(d, ak + 16, sdesc_advance(bk, 64), idesc, 1u);
            mma_f16_ts(d, ak + 24, sdesc_advance(bk, 96), idesc, 1u);
            mma_commit(stage_empty(cq.slot));
          }
          if (ok) mma_commit(tfull(tb));
        } else {
          for (int kb = w.kb0; kb < w.kb1; ++kb, cq.next(nslots)) {
            if (!(idle ? wait_sleepy(stage_full(cq.slot), cq.phase, abort_flag, args.status)
                       : wait_fast(stage_full(cq.slot), cq.phase, abort_flag, args.status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (!idle) {
              const uint64_t b0 = sdesc_sw128(x_stage(cq.slot));
              const uint64_t b1 = sdesc_advance(b0, box_rows * 128u);
              const uint32_t a0 = tmem_base + a_col + (uint32_t)cq.slot * 128u + mt * 64u;
              mma_f16_ts(d, a0, b0, idesc, kb == w.kb0 ? 0u : 1u);
              mma_f16_ts(d, a0 + 8, sdesc_advance(b0, 32), idesc, 1u);
              mma_f16_ts(d, a0 + 16, sdesc_advance(b0, 64), idesc, 1u);
              mma_f16_ts(d, a0 + 24, sdesc_advance(b0, 96), idesc, 1u);
              mma_f16_ts(d, a0 + 32, b1, idesc, 1u);
              mma_f16_ts(d, a0 + 40, sdesc_advance(b1, 32), idesc, 1u);
              mma_f16_ts(d, a0 + 48, sdesc_advance(b1, 64), idesc, 1u);
              mma_f16_ts(d, a0 + 56, sdesc_advance(b1, 96), idesc, 1u);
              mma_commit(stage_empty(cq.slot));
            } else {
              // nothing of this unit to track (its earlier MMAs completed before this
              // unit's accumulator barrier): a plain arrival, no tcgen05 instruction
              mbar_arrive(stage_empty(cq.slot));
            }
          }
          if (ok) {
            if (idle)
              mbar_arrive(tfull(tb));
            else
              mma_commit(tfull(tb));
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ unit scheduler
    // The global reads of a unit (its row block's expert segment, expert, real rows and the
    // expert's weight scale) happen here, up to kF4UnitRing units ahead of the other roles.
    if (lane == 0) {
      RingPos q{0, 0};
      for (int u = blockIdx.x; u < sched.units; u += gridDim.x, q.next(kF4UnitRing)) {
        const F4Desc d = f4_desc(args, sched, u, un);
        if (!wait_fast(unit_empty(q.slot), q.phase ^ 1u, abort_flag, args.status)) break;
        descs[q.slot] = d;
        mbar_arrive(unit_full(q.slot));
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + kF4CvtWarps) {
    // ------------------------------------------------------------ fp4 -> f16 into TMEM
    // Two groups of 8 converter warps take alternate stages, so that one group's load ->
    // convert -> TMEM store chain overlaps the other's (measured 2-3 % faster than all 16
    // warps on every stage). Warp c (0..15) of group c / 8 writes TMEM lane quarter c % 4
    // (= warp % 4, the quarter a warp may access): weight row 32 (c % 4) + lane of tile
    // (c / 4) % 2, both K chunks of the stage (64 values each: codes and four block
    // scales), i.e. that tile's 64 columns of the stage's A slot.
    const int c = warp - 4;
    const uint32_t grp = (uint32_t)(c >> 3);
    const int tile = (c >> 2) & 1;
    const uint32_t rr = (uint32_t)(32 * (c & 3) + lane);
    const bool live = tile < chunks;  // warp-uniform
    const uint32_t lanes = (uint32_t)(32 * (c & 3)) << 16;
    const uint32_t col0 = a_col + (uint32_t)tile * 64u;
    const uint32_t piece = (uint32_t)tile * kF4Piece;
    RingPos uq{0, 0}, rq{0, 0}, cq{0, 0};
    uint32_t jc = 0;  // stage counter of the CTA (both groups count every stage)
    bool ok = true;
    for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
      F4Desc w;
      if (!get_unit(uq, w)) break;
      release_unit(uq);
      for (int kb = w.kb0; kb < w.kb1;
           ++kb, ++jc, rq.next(kF4RawStages), cq.next(nslots)) {
        if ((jc & 1u) != grp) continue;
        if (!wait_fast(raw_full(rq.slot), rq.phase, abort_flag, args.status)) {
          ok = false;
          break;
        }
        const uint32_t src = raw_base + rq.slot * kF4RawBytes + piece;
        uint4 q0[2], q1[2];
        uint32_t scw[2] = {0u, 0u};
#pragma unroll
        for (int kc = 0; kc < 2; ++kc) {
          q0[kc] = make_uint4(0u, 0u, 0u, 0u);
          q1[kc] = q0[kc];
          if (live) {
            const uint32_t chunk = src + (uint32_t)kc * kFp4ChunkBytes;
            q0[kc] = lds128(chunk + rr * 16u);              // values 0..31 of the chunk
            q1[kc] = lds128(chunk + rr * 16u + 2048u);      // values 32..63
            scw[kc] = lds32(chunk + 4096u + rr * 4u);       // its four block scales
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty(rq.slot));
        if (!wait_fast(stage_empty(cq.slot), cq.phase ^ 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (live) {
#pragma unroll
          for (int kc = 0; kc < 2; ++kc) {
            uint32_t s0, s1, s2, s3;        // the block scales as f16 pairs
            e4m3x2_pairs(scw[kc] & 0xFFFFu, s0, s1);
            e4m3x2_pairs(scw[kc] >> 16, s2, s3);
            uint32_t o[32];
            const uint32_t words[8] = {q0[kc].x, q0[kc].y, q0[kc].z, q0[kc].w,
                                       q1[kc].x, q1[kc].y, q1[kc].z, q1[kc].w};
            const uint32_t scs[4] = {s0, s1, s2, s3};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t o4[4];
              e2m1x8_scaled(words[i], scs[i >> 1], o4);
              o[4 * i] = o4[0];
              o[4 * i + 1] = o4[1];
              o[4 * i + 2] = o4[2];
              o[4 * i + 3] = o4[3];
            }
            tmem_st32(tmem_base + lanes + col0 + (uint32_t)kc * 32u + (uint32_t)cq.slot * 128u,
                      o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(stage_full(cq.slot));
      }
    }
  } else if (warp >= 4 + kF4CvtWarps && warp < 4 + kF4CvtWarps + kF4EpiWarps) {
    // ------------------------------------------------------------ epilogue
    // D of tile t: TMEM lane = weight row (this warp's quarter), column j = the unit's token
    // row j. Lane l resolves token rows l, l + 32, l + 64, l + 96 to an output row and a
    // scale; every column is then one coalesced 128-byte store per warp.
    const int quarter = warp & 3;
    RingPos uq{0, 0};
    uint32_t uc = 0;
    for (int u = blockIdx.x; u < sched.units; u += gridDim.x, ++uc) {
      F4Desc w;
      if (!get_unit(uq, w)) break;
      release_unit(uq);
      const GemmProblem& P = args.p[w.p];
      const int tb = nbuf == 2 ? (int)(uc & 1u) : 0;   // accumulator buffer
      const uint32_t tph = nbuf == 2 ? ((uc >> 1) & 1u) : (uc & 1u);
      float* rowp[4] = {nullptr, nullptr, nullptr, nullptr};
      float rows_scale[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = lane + 32 * i;
        if (m >= w.rows) continue;
        const int mr = w.mb * kFp4BS + m;
        int f = -1;
        if (P.sorted_ids) {
          const int x = P.sorted_ids[mr];
          if (x >= 0 && x < P.num_flat) f = x;
        } else if (mr < P.store_rows) {
          f = mr;
        }
        if (f < 0) continue;
        float scale = w.alpha;
        float* out;
        if (KIND == kGemmW13) {
          out = P.part + (size_t)w.split * P.part_split_stride + (size_t)f * 2 * P.ldo;
        } else {
          int dest;
          if (P.sorted_ids) {
            dest = (f / P.top_k) * P.slots + (f % P.top_k);
            if (P.row_weight) scale = w.alpha * P.row_weight[f];
          } else {
            dest = f * P.slots + P.slot_offset;
          }
          out = static_cast<float*>(P.out) + (size_t)w.split * P.out_split_stride +
                (size_t)dest * P.ldo;
        }
        rowp[i] = out + (size_t)w.nt * un;
        rows_scale[i] = scale;
      }
      if (!wait_fast(tfull(tb), tph, abort_flag, args.status)) break;
      tc_fence_after();
      for (int t = 0; t < chunks; ++t) {
        const int col = t * kF4TileRows + 32 * quarter + lane;  // this lane's output column
        for (int c0 = 0; c0 < w.n; c0 += 16) {
          // tile t's accumulators in buffer tb: the two K chunks' (added in order), or,
          // for a unit of more than 64 rows, the one 128-column accumulator (its row half
          // holding columns c0 .. c0 + 15)
          const bool halves = w.n > 64;
          const int h = halves && c0 >= 64 ? 1 : 0;
          const uint32_t acc0 = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                ((uint32_t)tb * 4u + (uint32_t)(2 * t + h)) * acc_stride +
                                (uint32_t)(c0 - 64 * h);
          uint32_t v[16];
          tmem_ld16(acc0, v);
          tmem_wait_ld16(v);
          if (!halves) {
            uint32_t v2[16];
            tmem_ld16(acc0 + acc_stride, v2);
            tmem_wait_ld16(v2);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(v2[i]));
          }
          // the 32-row group of columns c0 .. c0 + 15 (warp-uniform)
          const int g = c0 >> 5;
          float* const gp = g == 0 ? rowp[0] : g == 1 ? rowp[1] : g == 2 ? rowp[2] : rowp[3];
          const float gs = g == 0 ? rows_scale[0]
                           : g == 1 ? rows_scale[1]
                           : g == 2 ? rows_scale[2] : rows_scale[3];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = c0 + i;  // token row of the unit (warp-uniform)
            if (j >= w.rows) break;
            float* const op = reinterpret_cast<float*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(gp), j & 31));
            const float sc = __shfl_sync(0xffffffffu, gs, j & 31);
            if (op) op[col] = sc * __uint_as_float(v[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(tb));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kF4TmemCols);
  }
}

template <int KIND>
cudaError_t launch_fp4_typed(const F4Maps& maps, const GemmLaunch& args, int grid,
                             cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_fp4_kernel<KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kF4Smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_kernel(gemm_fp4_kernel<KIND>, dim3(grid), dim3(kF4Threads), kF4Smem, stream,
                       maps, args);
}

}  // namespace

cudaError_t launch_gemm_fp4(int kind, const GemmLaunch& L, cudaStream_t stream) {
  if (L.num_problems < 1 || L.num_problems > 2 || L.splits < 1) return cudaErrorInvalidValue;
  if (kind != kGemmW13 && kind != kGemmW2) return cudaErrorInvalidValue;
  F4Maps maps;
  long units = 0;
  int max_box = 0;  // widest token box any unit of the launch can take
  // 256 weight rows per unit when every problem's weight rows split into 256s
  maps.un = kF4MaxN;
  for (int p = 0; p < L.num_problems; ++p)
    if (L.p[p].b_rows_per_expert % kF4MaxN) maps.un = kF4TileRows;
  // the caller counts K in 64-value chunks; the kernel's stages take two
  GemmLaunch Ls = L;
  for (int p = 0; p < 2; ++p) {
    const GemmProblem& P = L.p[L.num_problems > p ? p : 0];
    if (P.K % kF4StageK || P.k_blocks != P.K / kF4BK || P.b_rows_per_expert % maps.un ||
        P.n_tiles * maps.un != P.b_rows_per_expert || !P.B || !(P.gscale > 0.f) ||
        (reinterpret_cast<uintptr_t>(P.B) & 15u) || (kind == kGemmW13 ? !P.part : !P.out) ||
        P.ldo % 4)
      return cudaErrorInvalidValue;
    for (int i = 0; i < kF4Boxes; ++i)
      if (!make_map_2d(&maps.x[p][i], P.A, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)P.K,
                       (uint64_t)P.a_rows, (uint32_t)(16 << i)))
        return cudaErrorInvalidValue;
    if (p < L.num_problems) {
      Ls.p[p].k_blocks = P.K / kF4StageK;
      if (splits_of(L, p) < 1 || Ls.p[p].k_blocks < splits_of(L, p)) return cudaErrorInvalidValue;
      units += (long)P.max_m_blocks * P.n_tiles * splits_of(L, p);
      // an upper bound on the rows f4_desc gives a unit: routed blocks hold at most
      // rows_bound real rows; identity rows up to a block
      int rows = P.sorted_ids ? (P.rows_bound > 0 ? P.rows_bound : kFp4BS) : kFp4BS;
      if (!P.sorted_ids && P.store_rows < rows) rows = P.store_rows;
      rows = rows < 1 ? 1 : (rows > kFp4BS ? kFp4BS : rows);
      const int n = (rows + 15) & ~15;
      const int box = n <= 16 ? 0 : (n <= 32 ? 1 : (n <= 64 ? 2 : 3));
      if (box > max_box) max_box = box;
    }
  }
  // the token ring: per stage two boxes of the widest box, as many stages as the TMEM A ring
  maps.box_rows = 16 << max_box;
  maps.acc_stride = f4_acc(maps.box_rows);
  maps.tok_slot_bytes = 2 * maps.box_rows * 128;
  maps.slots = f4_slots(maps.box_rows);
  if (maps.slots * maps.tok_slot_bytes > (int)kF4TokArea) return cudaErrorInvalidValue;
  int grid = num_sms();
  if (units < grid) grid = (int)units;
  if (grid < 1) grid = 1;
  return kind == kGemmW13 ? launch_fp4_typed<kGemmW13>(maps, Ls, grid, stream)
                          : launch_fp4_typed<kGemmW2>(maps, Ls, grid, stream);
}

}  // namespace gbmoe
