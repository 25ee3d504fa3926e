// kda_chunk_tc.cu -- fused tensor-core chunked KDA forward for sm_103a (bf16 I/O,
// K = V = 128, chunk C = 64), one thread-block cluster per (sequence, value head).
//
// Chunked evaluation (page "手撕KDA", section "1 Naive", naive_chunk_kda; the
// decayed-operand factorisation follows the FlashKDA walk-through, page
// "KDA源码剖析之FlashKDA（上）", parts 9-11):
//   gc   = inclusive cumsum of g over the chunk rows, g_last = gc[C-1]
//   kd   = k e^{gc},  ki = k e^{-gc},  kr = k e^{g_last - gc},  qd = scale q e^{gc}
//   M    = strict_tril(Diag(beta) kd ki^T)        (beta scales rows)
//   Aqk  = tril(qd ki^T)                           (diagonal kept)
//   A    = (I + M)^{-1} Diag(beta)                 (beta scales columns)
//   W = A kd,  U = A v
//   per chunk, serially:  v_new = U - W S;  o = qd S + Aqk v_new;
//                         S <- Diag(e^{g_last}) S + kr^T v_new
//
// Work split.  The cluster's 4 CTAs each own a 32-column slice of V (the chain)
// and CTA r prepares the chunks n = r (mod 4) (the producer), so the
// V-independent preparation is done once per chunk.  A producer writes the
// chunk's record (qd, W, kr^T, Aqk in 128-byte-swizzled tile layout, U as four
// 32-column slices, e^{g_last}) into a per-head ring of 8 slots in the
// workspace (L2-resident; every part is staged in shared memory and written
// with bulk copies) and publishes it with a cluster-scope mbarrier arrive on
// every CTA; each CTA's chain bulk-copies the record into one of two
// shared-memory slots and acknowledges it back to the producer.  A producer
// keeps at most two records unacknowledged.  (Distributed shared memory
// measured ~17 B/clk per SM on GB300, too slow to carry ~60 KB per chunk; bulk
// copies from L2 are not.)
//
// Warps 0-3: producer.  Warps 4-7: chain (thread d holds row d of the fp32
// K x 32 state slice in registers; its bf16 copy in shared memory is the MMA
// operand; one chain thread also issues the record loads).  All dense
// contractions are tcgen05.mma with fp32 accumulators in TMEM:
//   producer: L = kd ki^T, Aqk = qd ki^T          (M=64, N=64,  K=128)
//             W = A kd, U = A v (B MN-major)       (M=64, N=128, K=64) x 2
//   chain:    X = W S, O = qd S                    (M=64, N=32,  K=128)
//             P = kr^T v_new                       (M=128,N=32,  K=64)
//             O += Aqk v_new                       (M=64, N=32,  K=64)
// The 64 x 64 unit-lower-triangular inverse runs on CUDA cores in fp32.
// Every wait is bounded; on a timeout a role records kStatusTimeout, all of
// its threads agree through bar.red.or, drain what they issued and return.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kda_common.cuh"
#include "sm103.cuh"

namespace kda {
namespace tc {

constexpr int C = 64;         // chunk rows
constexpr int KD = 128;       // key dim
constexpr int VD = 128;       // value dim
constexpr int VS = 32;        // value columns per CTA
constexpr int NSLICE = VD / VS;
constexpr int NTHREADS = 384; // 8 producer warps, 4 chain warps
constexpr uint32_t NPROD = 256, NCHAIN = 128;
constexpr int MB_LD = 68;     // padded row stride (floats) of the fp32 inverse buffer
constexpr int RING = 16;      // record slots per head in the workspace ring

// ---- record layout (global ring slot and shared slot share the first part) ----
// [W; qd] as one 128-row K-major operand: per 64-column K-block kb, W's 64
// rows (8 KB) then qd's 64 rows (8 KB), so X = W S and qd S are one M=128 MMA.
constexpr uint32_t R_WQ = 0;          // 2 K-blocks x [W rows | qd rows] bf16 SW128
constexpr uint32_t R_W_KB = 16384;    // stride between the K-blocks
constexpr uint32_t R_QD_IN_KB = 8192; // qd rows inside a K-block
constexpr uint32_t R_KRT = 32768;     // [128 x 64] bf16 SW128 (kr transposed)
constexpr uint32_t R_AQK = 49152;     // [64 x 64]  bf16 SW128, right after kr^T rows 64..127
constexpr uint32_t R_TILES = 57344;   // bytes of the tiles above
constexpr uint32_t G_U = 57344;       // global: 4 slices of U, each [64 x 32] bf16 row-major
constexpr uint32_t G_GAM = 57344 + 4 * 4096;  // global: e^{g_last} [128] fp32
constexpr uint32_t GSLOT = 74752;             // global slot stride (1024-multiple)
constexpr uint32_t S_U = 57344;       // shared slot: this CTA's U slice [64 x 32] bf16 row-major, replaced in
                                      // place by v_new (same 64 B per row, MN-major 64-byte swizzle)
constexpr uint32_t S_GAM = 61440;     // shared slot: e^{g_last} [128] fp32
constexpr uint32_t SSLOT = 62464;     // shared slot stride (1024-multiple)
constexpr uint32_t REC_TX = R_TILES + 4096 + 512;

// ---- shared memory map (offsets from a 1024-aligned base) ----
constexpr uint32_t OFF_SLOT = 0;                          // 2 record slots (chain)
constexpr uint32_t OFF_PREP = 2 * SSLOT;                  // 124928 producer tiles (prep:: layout)
constexpr uint32_t OFF_ST = OFF_PREP + 90112;             // 215040 S  [128 x 32] bf16 MN-major SW64 (chain)
constexpr uint32_t OFF_BETA = OFF_ST + 8192;              // 223232 [64] fp32
constexpr uint32_t OFF_GSUM = OFF_BETA + 256;             // 223488 [4][128] fp32 quarter-chunk sums of g
constexpr uint32_t OFF_RN = OFF_GSUM + 2048;              // 225536 [128] fp32 row norms of the raw q, k (pre-stage)
constexpr uint32_t OFF_BAR = OFF_RN + 512;                // 226048 mbarriers
constexpr uint32_t OFF_MISC = OFF_BAR + 256;              // 226304 tmem base
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;        // + alignment slack
static_assert(OFF_PREP % 1024 == 0 && SMEM_ALLOC <= 232448, "cluster kernel shared memory");

// barrier slots
constexpr int B_FULL = 0;    // [2] record landed in shared slot s (tx)
constexpr int B_PUB = 2;     // [4 x 2] record j of producer r published: index 2r + (j & 1) (remote arrive)
constexpr int B_ACK = 10;    // [2] this CTA's record j loaded by all 4 CTAs: index j & 1 (4 remote arrives)
constexpr int B_RAW = 12;    // producer raw q/k/v (tx)
constexpr int B_PMMA = 13;   // producer MMA commits
constexpr int B_A = 14;      // chain X/O MMA commit
constexpr int B_B = 15;      // chain P MMA commit
constexpr int B_C = 16;      // chain O += Aqk v_new commit

// TMEM columns
// chain: D_A[m & 1] holds X = W S in lanes 0-63 and o (qd S + Aqk v_new) in lanes
// 64-127, double-buffered across chunks; P = kr^T v_new
constexpr uint32_t TM_L = 0, TM_AQ = 64, TM_W = 0, TM_U = 128, TM_A0 = 256, TM_P = 320;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t RAW_TX_BYTES = 3 * 16384;        // q, k, v tiles
// Bounded waits.  A wait for work (a record, a flag, a product or tile this role has not
// seen complete yet) gives up after p.wait_ns (2 s unless the caller's environment
// sets KDA_WAIT_LIMIT_NS); a drain wait (for copies and products already issued, before
// the block reuses or releases the memory they touch) always allows DRAIN_LIMIT_NS.
constexpr uint64_t DRAIN_LIMIT_NS = 2000000000ull;   // 2 s

constexpr uint32_t NB_PREP = 1, NB_CHAIN = 2;

struct Maps {
  CUtensorMap q32, k32;  // q, k with 32-token boxes (the stacked producer tile)
  CUtensorMap v;         // v with 64-token boxes
  CUtensorMap o;         // output tiles (split kernel)
};

// Optional instrumentation (build with -DKDA_PROFILE), stored as uint64 words after
// the status word of the workspace: per-phase clock64 sums of one producer and one
// chain thread of the cluster kernel ([1, 17) and [17, 33)); in the split kernel, for
// unit 0, the globaltimer stamps of each record's publication [200, 264), of its two
// copies' issue [264, 328) and [330, 394) and of the chain's start [127], the clock64
// stamps of threads 0 and 256 at the numbered points of one chunk [432, 480), and
// [400] the first timeout (block << 40 | thread << 24 | chunk << 8 | wait site).
#ifdef KDA_PROFILE
#define PROF_DECL                                 \
  uint64_t prof_acc[16] = {0};                    \
  uint64_t prof_last = clock64();                 \
  const bool prof_on = (blockIdx.x | blockIdx.y | blockIdx.z) == 0;
#define PROF(i)                                 \
  do {                                          \
    if (prof_on) {                              \
      const uint64_t t_ = clock64();            \
      prof_acc[i] += t_ - prof_last;            \
      prof_last = t_;                           \
    }                                           \
  } while (0)
#define PROF_STORE(base)                                                            \
  do {                                                                              \
    if (prof_on) {                                                                  \
      uint64_t* dst_ = reinterpret_cast<uint64_t*>(p.status) + 1 + (base);          \
      for (int i_ = 0; i_ < 16; ++i_) dst_[i_] = prof_acc[i_];                      \
    }                                                                               \
  } while (0)
#else
#define PROF_DECL
#define PROF(i) \
  do {          \
  } while (0)
#define PROF_STORE(base) \
  do {                   \
  } while (0)
#endif

constexpr float kLog2e = 1.4426950408889634f;
// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLn2 = 0.6931471805599453f;
__device__ __forceinline__ float rcp_approx(float x) {  // 1 / x (PTX rcp.approx; 1 / inf = 0)
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sigmoid(x) = 1 / (1 + e^-x) = (1 + tanh(x / 2)) / 2: one special-function instruction
__device__ __forceinline__ float sigmoid_approx(float x) { return fmaf(0.5f, tanh_approx(0.5f * x), 0.5f); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
// two floats -> bf16 pair (lo in the low half), one paired conversion instruction
// (float -> bf16 conversions issue at a fraction of the FMA rate)
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void st_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}
__device__ __forceinline__ void st_v4_global(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  __stcg(reinterpret_cast<uint4*>(p), make_uint4(a, b, c, d));
}

// Role barriers: reconverge the warp first (bar.sync / bar.red are .aligned).
__device__ __forceinline__ void role_sync(uint32_t id, uint32_t count) {
  __syncwarp();
  named_bar_sync(id, count);
}
__device__ __forceinline__ bool role_any(uint32_t id, uint32_t count, bool pred) {
  __syncwarp();
  return named_bar_any(id, count, pred);
}

// Off-diagonal blocks of T = (I + M)^{-1} (64 x 64, 16 x 16 blocks), given the
// inverted diagonal blocks T_ii on the diagonal of `mb` and M below it.  Warp w
// (0..2) walks block column w down its block rows i > w, in transposed form:
//     R^T = sum_{k = w}^{i-1} T_kw^T M_ik^T,    T_iw^T = -R^T T_ii^T,
// as m16n8k8 TF32 MMAs (operands truncated to TF32, fp32 accumulation).  Block
// column w needs only itself and the diagonal blocks, so the warps never wait on
// one another.  R^T stays in registers: the accumulator of n-tile nt is the A
// operand of k-step nt once the k index inside a step is read in the order
// 0, 2, 4, 6, 1, 3, 5, 7 (thread (g, t) holds columns 2t and 2t + 1), so the B
// operand rows are taken in that order too.  T_iw is kept transposed in the
// unused block (w, i) above the diagonal (mb[16 w + col][16 i + row]), from where
// it is the next A operand, and written, scaled by beta of its column, into the
// bf16 A tile.  The block column is a template argument so that every loop is
// unrolled and the operand loads of a step are issued ahead of its MMAs (a
// run-time block column measured 2.4x slower).
template <int w>
__device__ __forceinline__ void inverse_block_column(float* mb, const float* beta_s, uint8_t* amat, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = w + 1; i < 4; ++i) {
    float r[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // R^T, n-tile nt: rows 8 nt + [0, 8) of block i
#pragma unroll
    for (int k = w; k < i; ++k) {
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4];  // A = T_kw^T: m = column in block column w, kk = row in block k
        if (k == w) {   // T_ww, row-major on the diagonal
          const float* pa = mb + (16 * w + 8 * ks + t) * MB_LD + 16 * w + g;
          a[0] = __float_as_uint(pa[0]);
          a[1] = __float_as_uint(pa[8]);
          a[2] = __float_as_uint(pa[4 * MB_LD]);
          a[3] = __float_as_uint(pa[4 * MB_LD + 8]);
        } else {  // T_kw, transposed in block (w, k)
          const float* pa = mb + (16 * w + g) * MB_LD + 16 * k + 8 * ks + t;
          a[0] = __float_as_uint(pa[0]);
          a[1] = __float_as_uint(pa[8 * MB_LD]);
          a[2] = __float_as_uint(pa[4]);
          a[3] = __float_as_uint(pa[8 * MB_LD + 4]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {  // B = M_ik^T
          const float* pb = mb + (16 * i + 8 * nt + g) * MB_LD + 16 * k + 8 * ks + t;
          mma_tf32_m16n8k8(r[nt], a, __float_as_uint(pb[0]), __float_as_uint(pb[4]));
        }
      }
    }
    float tv[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // -T_iw^T
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const uint32_t a[4] = {__float_as_uint(r[ks][0]), __float_as_uint(r[ks][2]), __float_as_uint(r[ks][1]),
                             __float_as_uint(r[ks][3])};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {  // B = T_ii^T, rows 8 ks + 2t and 8 ks + 2t + 1
        const float2 b = *reinterpret_cast<const float2*>(mb + (16 * i + 8 * nt + g) * MB_LD + 16 * i + 8 * ks + 2 * t);
        mma_tf32_m16n8k8(tv[nt], a, __float_as_uint(b.x), __float_as_uint(b.y));
      }
    }
    // tv[nt][e] = -T_iw[8 nt + 2t + (e & 1)][g + 8 (e >> 1)]
    const float bl = beta_s[16 * w + g], bh = beta_s[16 * w + g + 8];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int row = 8 * nt + 2 * t;
      *reinterpret_cast<float2*>(mb + (16 * w + g) * MB_LD + 16 * i + row) = make_float2(-tv[nt][0], -tv[nt][1]);
      *reinterpret_cast<float2*>(mb + (16 * w + g + 8) * MB_LD + 16 * i + row) = make_float2(-tv[nt][2], -tv[nt][3]);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        *reinterpret_cast<uint16_t*>(amat + sw128_offset(16 * i + row + e, 16 * w + g, 64)) = f2bf(-tv[nt][e] * bl);
        *reinterpret_cast<uint16_t*>(amat + sw128_offset(16 * i + row + e, 16 * w + g + 8, 64)) =
            f2bf(-tv[nt][2 + e] * bh);
      }
    }
    __syncwarp();  // T_iw visible to this warp's later block rows
  }
}
__device__ __forceinline__ void inverse_block_columns(float* mb, const float* beta_s, uint8_t* amat, int w, int lane) {
  if (w == 0) inverse_block_column<0>(mb, beta_s, amat, lane);
  else if (w == 1) inverse_block_column<1>(mb, beta_s, amat, lane);
  else if (w == 2) inverse_block_column<2>(mb, beta_s, amat, lane);
}

// ======================================================================
// Chunk preparation shared by both kernels' producers: the decayed operands, the
// products L = kd ki^T and Aqk = qd ki^T, and their readout.
//
// Range.  A factorisation e^{gc_i - gc_j} = e^{gc_i - r} e^{r - gc_j} is exact only
// while both factors are representable.  With one reference r per chunk (the chunk
// start) e^{-gc_j} overflows once a chunk's cumulative decay passes about -88, which
// the bounded gate of the method (g >= -5 per token, i.e. -320 over 64 tokens) reaches
// easily.  So the lower triangles of L and Aqk are formed as three blocks:
//   * the two 32 x 32 diagonal halves, each referenced at its middle row (the end of
//     its first 16-row quarter): every factor is bounded by the decay over 16 tokens;
//   * the 32 x 32 block below them (rows 32-63, columns 0-31), whose rows reuse the
//     second half's operands (reference: row 48) and whose columns carry
//     e^{gc_47 - gc_j} <= 1.  A column factor that flushes to zero (below 2^-126)
//     drops a product smaller than 2^{-126} times the row factor, itself at most
//     2^{-s_2} (s_2 the decay of rows 32-47, log2 units), so under the range below the
//     dropped terms are under 2^-10, beneath the bf16 rounding of the operands.
// The factors are built from the within-quarter cumsum x (0 >= x >= s_q, the quarter's
// decay in log2 units) and per-quarter constants, so no intermediate leaves the range
// either.  The supported range is therefore: the decay of every 16-token quarter of a
// chunk (per key dimension) is >= kMinQuarterLog2 = -116 (-80.4 in natural-log
// units), which g >= -5 per token meets; the producers report a quarter outside it
// with kStatusRange.  The chunk-start-referenced factors kd, qd and kr are all <= 1
// (their underflow is harmless) and stay as they were.
//
// Tile layout of a producer (offsets from its 1024-aligned base; bf16 K-major tiles in
// the 128-byte swizzle layout, two 64-column K-blocks each):
//   QK    stacked [k rows 0-31 | q rows 0-31 | k rows 32-63 | q rows 32-63], the raw tiles
//         as TMA lands them (32-row boxes), rewritten in place as kA / qA (half-middle
//         reference): the 128-row A operand of the L/Aqk product
//   CC    [cA rows 0-63 | cB rows 0-31]: its 96-row B operand, cA = k e^{mid - gc}
//         (reference: the row's own half) and cB = k e^{gc_47 - gc} (rows of the first half)
//   KDT   kd = k e^{gc} (64 rows): MN-major B operand of W = A kd
//   VRAW  the raw v tiles (loaded with q and k)
//   QDS   (split kernel) qd staging, bulk-copied into the record
// and, once the products have read them,
//   MB / AMAT  M (fp32) and A = T Diag(beta) (bf16) over QK;  AQK_STG (bf16 Aqk) and
//   then the U staging over CC;  the W staging over KDT.
// kr^T (and, in the cluster kernel, qd) is written by the elementwise pass straight into the
// record (global).
// ======================================================================
namespace prep {
constexpr uint32_t QK = 0;
constexpr uint32_t QK_KB = 16384;  // one K-block of the stacked 128-row tile
constexpr uint32_t CC = 32768;     // [cA rows 0-63 | cB rows 0-31]: the 96-row B operand
constexpr uint32_t CC_KB = 12288;  // one K-block of it
constexpr uint32_t KDT = 57344;
constexpr uint32_t VRAW = 73728;
constexpr uint32_t BYTES = 90112;
constexpr uint32_t QDS = BYTES;        // optional qd staging tile (64 rows), right after the others
constexpr uint32_t MB = QK;
constexpr uint32_t AMAT = QK + 17408;  // after M (64 x MB_LD fp32)
constexpr uint32_t AQK_STG = CC;
constexpr uint32_t USTG = CC;          // after the Aqk staging has been read
static_assert(AMAT + 8192 <= CC && MB_LD * 64 * 4 <= 17408, "M and A fit the stacked tile");
static_assert(CC + 2 * CC_KB <= KDT && KDT + 16384 <= VRAW && VRAW + 16384 <= BYTES, "producer tiles");
constexpr uint32_t RAW_TX = 32768 + 16384;  // q, k and v tiles of one chunk
// TMEM columns of the L/Aqk product (relative to the producer's TMEM base): M = 128, N = 96,
// lane r = stacked row r; columns 0-63 against cA, 64-95 against cB
constexpr uint32_t TM_LQ = 0;
constexpr float kMinQuarterLog2 = -116.f;

// q, k (into the stacked tile, 32-row boxes) and v tiles of chunk rows [row0, row0 + 64).
__device__ __forceinline__ void issue_raw(uint8_t* base, const CUtensorMap* q32, const CUtensorMap* k32,
                                          const CUtensorMap* v, uint64_t* bar, int hk, int hv, int row0) {
  mbar_arrive_expect_tx(bar, RAW_TX);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    uint8_t* t = base + QK + kb * QK_KB;
    tma_load_3d(t, k32, bar, 64 * kb, hk, row0);
    tma_load_3d(t + 4096, q32, bar, 64 * kb, hk, row0);
    tma_load_3d(t + 8192, k32, bar, 64 * kb, hk, row0 + 32);
    tma_load_3d(t + 12288, q32, bar, 64 * kb, hk, row0 + 32);
  }
  tma_load_3d(base + VRAW, v, bar, 0, hv, row0);
  tma_load_3d(base + VRAW + 8192, v, bar, 64, hv, row0);
}

// Two fp32 lanes in one 64-bit register: the packed (.f32x2) multiply of sm_100 and later
// does both dims of a thread in one instruction.
__device__ __forceinline__ unsigned long long f2u(float lo, float hi) {
  unsigned long long u;
  asm("mov.b64 %0, {%1, %2};" : "=l"(u) : "f"(lo), "f"(hi));
  return u;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// bf16 pair (lo in the low half) of a packed fp32 pair
__device__ __forceinline__ uint32_t pack2u(unsigned long long u) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(u));
  return pack2(lo, hi);
}
// the two fp32 values of a bf16 pair, as a packed fp32 pair
__device__ __forceinline__ unsigned long long bf2u(uint32_t b) {
  return f2u(__uint_as_float(b << 16), __uint_as_float(b & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Pre-stage of the gated forward, on the thread's 16 rows x 2 dims of raw gate input
// (g: raw values in, activated g out; rows past the end become 0) and, for the first
// 64 threads, its row's raw beta: the bounded gate lower_bound sigmoid(a (g + dt)) or
// the softplus gate -a softplus(g + dt), a = exp(A_log) of the value head, and beta =
// sigmoid(beta).  (Pages "手撕KDA" section 2 and "KDA源码剖析之FlashKDA（上）" part 7.)
__device__ __forceinline__ void activate(float2 (&g)[16], float& beta, int kind, float lb, float a, float2 dt,
                                         int hq, int pt, int rows) {
  const int nvalid = rows - 16 * hq;
  if (kind == 1) {  // lb sigmoid(a x) = lb/2 + (lb/2) tanh(a x / 2), a x / 2 = ha g + ha dt
    const float ha = 0.5f * a, hl = 0.5f * lb;
    const float hdx = ha * dt.x, hdy = ha * dt.y;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      g[i] = make_float2(fmaf(hl, tanh_approx(fmaf(ha, g[i].x, hdx)), hl),
                         fmaf(hl, tanh_approx(fmaf(ha, g[i].y, hdy)), hl));
    if (nvalid < 16) {  // a sequence's partial last chunk: rows past the end act as g = 0
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i >= nvalid) g[i] = make_float2(0.f, 0.f);
    }
  } else {
    auto softplus = [](float x) {  // log(1 + e^x), with its two asymptotes
      return x > 20.f ? x : (x < -20.f ? ex2_approx(x * kLog2e) : lg2_approx(1.f + ex2_approx(x * kLog2e)) * kLn2);
    };
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float x0 = -a * softplus(g[i].x + dt.x), x1 = -a * softplus(g[i].y + dt.y);
      g[i] = i < nvalid ? make_float2(x0, x1) : make_float2(0.f, 0.f);
    }
  }
  if (pt < C) beta = pt < rows ? sigmoid_approx(beta) : 0.f;
}

// The gate rows a thread prefetched (rows 16 hq + [0, 16), key dims 2 dp, 2 dp + 1) are
// loaded unconditionally from row min(c, rows - 1), so that no instruction waits for
// them before their first use: with PRE the raw bf16 pair sits in .x; rows past the end
// become 0, as does beta there.
template <bool PRE>
__device__ __forceinline__ void finish_gate_rows(float2 (&g)[16], float& beta, int hq, int pt, int rows) {
  const int nvalid = rows - 16 * hq;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (PRE) {
      const uint32_t w = __float_as_uint(g[i].x);
      g[i] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
    if (i >= nvalid) g[i] = make_float2(0.f, 0.f);
  }
  if (pt >= rows) beta = 0.f;
}

// 1 / sqrt(|row|^2 + 1e-6) of every row of the stacked raw tile (k and q rows), into
// rn[stacked row]: thread pt sums the squares of K-block pt & 1 of stacked row pt / 2,
// its neighbour lane the other K-block.
__device__ __forceinline__ void row_norms(const uint8_t* base, float* rn, int pt) {
  const int srow = pt >> 1, kb = pt & 1;
  const uint4* r = reinterpret_cast<const uint4*>(base + QK + kb * QK_KB + srow * 128);
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 u = r[c];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float lo = __uint_as_float(w[t] << 16), hi = __uint_as_float(w[t] & 0xFFFF0000u);
      ss = fmaf(lo, lo, fmaf(hi, hi, ss));
    }
  }
  ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
  if (kb == 0) rn[srow] = rsqrtf(ss + 1e-6f);
}

// Elementwise pass of thread (dp, hq): key dims 2 dp, 2 dp + 1 of chunk rows
// [16 hq, 16 hq + 16) (quarter hq).  gsum holds the four quarter sums of g (natural
// log) per key dim; g holds this thread's 16 rows.  Writes kA/qA (in place), cA, kd and
// (hq < 2) cB to the tiles, kr^T and (hq = 0) e^{g_last} into the record (krt_rec +
// SW128 offset in the [128 x 64] kr^T tile, gam_rec), and qd either to the tile QDS
// (QD_SMEM, for a bulk copy) or into the record (qd_rec + kb * qd_kb_stride + SW128 row
// offset); without KR, kr^T and e^{g_last} are not written.  With NORM, k and q rows are first scaled by their rn[] entries (the
// pre-stage's L2 normalisation).  Sets range_bad when this quarter decays faster
// than the factors can represent.
//
// With x the within-quarter cumsum (log2 units; 0 >= x >= sh, sh the quarter's sum),
// pre the decay before the quarter and all the chunk's:
//   kd, qd = (k, scale q) 2^pre 2^x            kr = k 2^{all - pre - sh} (2^sh 2^-x)
//   kA, qA = (k, scale q) 2^x (2^-sh if hq even: the half's middle is the quarter's end)
//   cA     = k 2^-x (2^sh if hq even)
//   cB     = k (2^sh 2^-x) 2^{s_2} (2^{s_1} if hq = 0)      [reference: row 48]
// where 2^sh 2^-x lies in [2^sh, 1] and every other product of factors is <= 1.
//
// Addressing: every tile base is 1024-aligned and a row is 128 bytes, so the 128-byte
// swizzle (16-byte chunk index XOR row % 8) is an XOR on address bits 4-6 that commutes
// with adding the row and the tile offsets; one 32-bit shared address per row serves
// all tiles.
template <bool QD_SMEM, bool NORM, bool KR = true>
__device__ __forceinline__ void elementwise(uint8_t* base, const float* gsum, const float2 (&g)[16], int dp, int hq,
                                            int rows, float scale, uint8_t* qd_rec, uint32_t qd_kb_stride,
                                            uint8_t* krt_rec, float* gam_rec, const float* rn, bool& range_bad) {
  float c_d[2], c_r[2], es[2], fa[2], fb[2];
  const bool even = (hq & 1) == 0;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float s[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) s[qq] = gsum[qq * tc::KD + 2 * dp + e] * kLog2e;
    const float all = (s[0] + s[1]) + (s[2] + s[3]);
    const float pre = hq == 0 ? 0.f : hq == 1 ? s[0] : hq == 2 ? s[0] + s[1] : (s[0] + s[1]) + s[2];
    const float sh = hq == 0 ? s[0] : hq == 1 ? s[1] : hq == 2 ? s[2] : s[3];
    if (!(sh >= kMinQuarterLog2)) range_bad = true;
    c_d[e] = ex2_approx(pre);
    c_r[e] = ex2_approx(all - pre - sh);
    es[e] = ex2_approx(sh);
    fa[e] = even ? ex2_approx(-sh) : 1.f;                       // kA, qA
    fb[e] = ex2_approx(hq == 0 ? s[1] + s[2] : s[2]);           // cB (hq < 2)
    if (KR && hq == 0) gam_rec[2 * dp + e] = ex2_approx(all);
  }
  // the per-dim constants as packed pairs
  const unsigned long long CD = f2u(c_d[0], c_d[1]), CR = f2u(c_r[0], c_r[1]), ES = f2u(es[0], es[1]),
                           FA = f2u(fa[0], fa[1]), FB = f2u(fb[0], fb[1]), SC = f2u(scale, scale);
  const uint32_t kb = static_cast<uint32_t>(dp) >> 5;
  const uint32_t r0 = 16u * static_cast<uint32_t>(hq);
  const uint32_t lo = ((2u * dp) & 7u) * 2u;
  const uint32_t c4 = (((2u * dp) & 63u) >> 3) << 4;  // unswizzled 16-byte chunk offset
  // row r0 of each tile, before the swizzle XOR (tile offsets and rows keep bits 4-6 clear)
  const uint32_t X = smem_u32(base) + r0 * 128u + lo + c4;
  const uint32_t a_k = QK + kb * QK_KB + (hq >= 2 ? 32u : 0u) * 128u;  // stacked row of k row r0
  const uint32_t a_c = CC + kb * CC_KB;                                // cA row r0 (cB: + 64 rows)
  const uint32_t a_d = KDT + kb * 8192u;                               // kd (and the qd staging: + QDS - KDT)
  uint8_t* qdr = qd_rec + kb * qd_kb_stride + r0 * 128u + lo;
  const int nvalid = rows - static_cast<int>(r0);  // rows of this quarter that exist (may be <= 0 or > 16)
  uint32_t kr[2][4];
  uint32_t kre = 0u;  // kr of the previous (even) row, bf16 pair (dims 2 dp, 2 dp + 1)
  float x0 = 0.f, x1 = 0.f;
  uint32_t kn = lds32(X + a_k), qn = lds32(X + a_k + 4096u);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t swz = (static_cast<uint32_t>(i) & 7u) << 4;
    const uint32_t Y = (X ^ swz) + static_cast<uint32_t>(i) * 128u;  // row r0 + i, any tile
    const uint32_t vm = i < nvalid ? 0xFFFFFFFFu : 0u;                // rows past the end act as k = q = 0
    const uint32_t kraw = kn & vm, qraw = qn & vm;
    if (i < 15) {  // the next row's raw values, ahead of this row's stores
      const uint32_t Yn = (X ^ ((static_cast<uint32_t>(i + 1) & 7u) << 4)) + static_cast<uint32_t>(i + 1) * 128u;
      kn = lds32(Yn + a_k);
      qn = lds32(Yn + a_k + 4096u);
    }
    x0 = fmaf(g[i].x, kLog2e, x0);
    x1 = fmaf(g[i].y, kLog2e, x1);
    const unsigned long long E = f2u(ex2_approx(x0), ex2_approx(x1));
    const unsigned long long IE = f2u(ex2_approx(-x0), ex2_approx(-x1));
    unsigned long long Kv = bf2u(kraw), Qv = mul2(bf2u(qraw), SC);
    if (NORM) {
      const uint32_t srow = (hq >= 2 ? 32u : 0u) + r0 + i;  // stacked row of k row r0 + i (q: + 32)
      const float rk = rn[srow], rq = rn[srow + 32];
      Kv = mul2(Kv, f2u(rk, rk));
      Qv = mul2(Qv, f2u(rq, rq));
    }
    const unsigned long long Pv = mul2(IE, ES);  // 2^{sh - x}
    {
      const unsigned long long Av = even ? mul2(E, FA) : E;
      sts32(Y + a_k, pack2u(mul2(Kv, Av)));
      sts32(Y + a_k + 4096u, pack2u(mul2(Qv, Av)));
      sts32(Y + a_c, pack2u(mul2(Kv, even ? Pv : IE)));
    }
    {
      const unsigned long long Dv = mul2(E, CD);
      sts32(Y + a_d, pack2u(mul2(Kv, Dv)));
      if (QD_SMEM)
        sts32(Y + a_d + (QDS - KDT), pack2u(mul2(Qv, Dv)));
      else
        __stcg(reinterpret_cast<uint32_t*>(qdr + ((c4 ^ swz) + static_cast<uint32_t>(i) * 128u)), pack2u(mul2(Qv, Dv)));
    }
    if (hq < 2) sts32(Y + a_c + 64u * 128u, pack2u(mul2(Kv, mul2(Pv, FB))));
    // kr^T rows 2 dp and 2 dp + 1: bf16 pairs along the tokens
    const uint32_t krp = pack2u(mul2(Kv, mul2(Pv, CR)));
    if (i & 1) {
      kr[0][(i >> 1) & 3] = __byte_perm(kre, krp, 0x5410);
      kr[1][(i >> 1) & 3] = __byte_perm(kre, krp, 0x7632);
    } else {
      kre = krp;
    }
    if (KR && (i & 7) == 7)  // tokens r0 + i - 7 .. r0 + i
#pragma unroll
      for (int e = 0; e < 2; ++e)
        __stcg(reinterpret_cast<uint4*>(krt_rec + sw128_offset(2 * dp + e, r0 + (i & 8), 128)),
               make_uint4(kr[e][0], kr[e][1], kr[e][2], kr[e][3]));
  }
}

// The L/Aqk product (issued by one converged warp): the stacked [kA; qA] rows (M = 128)
// against [cA; cB] (N = 96).  Columns 0-63 hold the diagonal halves of L and Aqk
// (rows and columns of the same half), columns 64-95 of lanes 64-127 the block below
// them (rows 32-63 of L and Aqk against columns 0-31).
__device__ __forceinline__ void issue_lqk(uint32_t tmem, uint64_t d_sw128) {
  auto d = [&](uint32_t off) { return d_sw128 + (off >> 4); };
  constexpr uint32_t idesc = idesc_f16kind(128, 96);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_f16_warp(tmem + TM_LQ, d(QK + kb * QK_KB + ks * 32), d(CC + kb * CC_KB + ks * 32), idesc, (kb | ks) != 0);
}

// Readout by the 8 warps of a producer (quad = TMEM lane quadrant = which 32 stacked
// rows, cpart = which 16 columns): M = strict_tril(Diag(beta) L) as fp32 into MB (the
// upper-right 32 x 32 block is not written: the inverse never reads it as M) and
// Aqk = tril(qd ki^T) as the bf16 SW128 tile AQK_STG (every element written).
__device__ __forceinline__ void readout_lqk(uint8_t* base, uint32_t tmem, const float* beta_s, int quad, int cpart,
                                            int lane) {
  float* mb = reinterpret_cast<float*>(base + MB);
  uint8_t* aq = base + AQK_STG;
  const int half = quad >> 1;
  const int i = 32 * half + lane;         // row of L (quad 0, 2) or Aqk (quad 1, 3)
  const int c0 = 32 * half + 16 * cpart;  // diagonal-half columns of this warp
  float dv[16], ov[16];
  tmem_ld16(tmem_addr(tmem, 32 * quad, TM_LQ + c0), dv);
  // columns 16 cpart + [0, 16) of the block below the halves (used by quadrants 2 and 3; the
  // load is unconditional, which keeps the compiler's register allocation simple)
  tmem_ld16(tmem_addr(tmem, 32 * quad, TM_LQ + 64 + 16 * cpart), ov);
  tmem_ld_wait();
  if ((quad & 1) == 0) {  // L
    const float bi = beta_s[i];
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      float4 v4;
      const int c = c0 + 4 * j4;
      v4.x = (c + 0 < i) ? bi * dv[4 * j4 + 0] : 0.f;
      v4.y = (c + 1 < i) ? bi * dv[4 * j4 + 1] : 0.f;
      v4.z = (c + 2 < i) ? bi * dv[4 * j4 + 2] : 0.f;
      v4.w = (c + 3 < i) ? bi * dv[4 * j4 + 3] : 0.f;
      *reinterpret_cast<float4*>(mb + i * MB_LD + c) = v4;
    }
    if (half)  // the block below the halves: no mask
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4)
        *reinterpret_cast<float4*>(mb + i * MB_LD + 16 * cpart + 4 * j4) =
            make_float4(bi * ov[4 * j4], bi * ov[4 * j4 + 1], bi * ov[4 * j4 + 2], bi * ov[4 * j4 + 3]);
  } else {  // Aqk (diagonal kept)
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
      uint32_t w[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int c = c0 + 8 * h8 + 2 * t;
        w[t] = pack2((c <= i) ? dv[8 * h8 + 2 * t] : 0.f, (c + 1 <= i) ? dv[8 * h8 + 2 * t + 1] : 0.f);
      }
      st_v4(aq + sw128_offset(i, c0 + 8 * h8, 64), w[0], w[1], w[2], w[3]);
    }
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
      if (half)  // rows 32-63, columns 0-31: the block below the halves
        st_v4(aq + sw128_offset(i, 16 * cpart + 8 * h8, 64), pack2(ov[8 * h8], ov[8 * h8 + 1]),
              pack2(ov[8 * h8 + 2], ov[8 * h8 + 3]), pack2(ov[8 * h8 + 4], ov[8 * h8 + 5]),
              pack2(ov[8 * h8 + 6], ov[8 * h8 + 7]));
      else  // rows 0-31, columns 32-63: zero
        st_v4(aq + sw128_offset(i, 32 + 16 * cpart + 8 * h8, 64), 0u, 0u, 0u, 0u);
    }
  }
}

// Diagonal 16 x 16 blocks of T = (I + M)^{-1} by forward substitution (warps 0-3, one
// column per lane of the first half-warp), written to MB and, scaled by beta of the
// column, to AMAT; warps 4-7 zero the blocks of AMAT above the diagonal.
__device__ __forceinline__ void inverse_diag_blocks(uint8_t* base, const float* beta_s, int pw, int pt, int lane) {
  float* mb = reinterpret_cast<float*>(base + MB);
  uint8_t* amat = base + AMAT;
  if (pw < 4) {
    if (lane < 16) {
      const int b0 = 16 * pw, jc = lane;
      // row by row: T[i][jc] = [i == jc] - sum_{mm < i} M[i][mm] T[mm][jc], with
      // M's row read four at a time and two partial sums
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float* row = mb + (b0 + i) * MB_LD + b0;
        float s0 = (i == jc) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
        for (int mm = 0; mm < i; mm += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(row + mm);
          s0 = fmaf(-m4.x, acc[mm], s0);
          if (mm + 1 < i) s1 = fmaf(-m4.y, acc[mm + 1], s1);
          if (mm + 2 < i) s0 = fmaf(-m4.z, acc[mm + 2], s0);
          if (mm + 3 < i) s1 = fmaf(-m4.w, acc[mm + 3], s1);
        }
        acc[i] = s0 + s1;
      }
      __syncwarp(0x0000FFFFu);
      const float bj = beta_s[b0 + jc];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        mb[(b0 + i) * MB_LD + b0 + jc] = acc[i];
        *reinterpret_cast<uint16_t*>(amat + sw128_offset(b0 + i, b0 + jc, 64)) = f2bf(acc[i] * bj);
      }
    }
  } else {
    // blocks (row block br, column block bc > br): 6 blocks of 16 x 16 bf16 zeros,
    // 2 chunks of 8 columns per row -> 6 * 16 * 2 = 192 16-byte stores over 128 threads
    for (int idx = pt - 128; idx < 192; idx += 128) {
      const int blk = idx >> 5, rem = idx & 31, row = rem >> 1, hf = rem & 1;
      const int br = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bc = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      st_v4(amat + sw128_offset(16 * br + row, 16 * bc + 8 * hf, 64), 0u, 0u, 0u, 0u);
    }
  }
}
}  // namespace prep

// PRE: the pre-stage of the gated forward is fused in (p.prestage != 0): raw bf16 gate
// input, beta sigmoid and q/k L2 normalisation (a separate instantiation, so that the
// plain forward carries none of it)
template <bool PRE>
__global__ void __cluster_dims__(NSLICE, 1, 1) __launch_bounds__(NTHREADS, 1)
kda_chunk_fused_kernel(const __grid_constant__ Maps maps, const FwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  float* beta_s = reinterpret_cast<float*>(sm + OFF_BETA);
  float* gsum = reinterpret_cast<float*>(sm + OFF_GSUM);
  float* rn = reinterpret_cast<float*>(sm + OFF_RN);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hv = blockIdx.y, seq = blockIdx.z;
#ifdef KDA_PROFILE
  const uint64_t kt0 = globaltimer_ns();
#endif
  const uint32_t rank = cluster_ctarank();  // == blockIdx.x: the V slice and producer index
  const int HV = p.HV;
  const int hk = hv / (HV / p.H);
  const int v0 = static_cast<int>(rank) * VS;

  long tok0;
  int len;
  seq_range(p, seq, tok0, len);
  const int NT = (len + C - 1) / C;
  uint8_t* ring = p.ring + (static_cast<size_t>(seq) * HV + hv) * (static_cast<size_t>(RING) * GSLOT);

  if (tid == 0) {
    mbar_init(&bars[B_FULL], 1);
    mbar_init(&bars[B_FULL + 1], 1);
    for (int r = 0; r < 8; ++r) mbar_init(&bars[B_PUB + r], 1);
    mbar_init(&bars[B_ACK], NSLICE);
    mbar_init(&bars[B_ACK + 1], NSLICE);
    mbar_init(&bars[B_RAW], 1);
    mbar_init(&bars[B_PMMA], 1);
    mbar_init(&bars[B_A], 1);
    mbar_init(&bars[B_B], 1);
    mbar_init(&bars[B_C], 1);
    fence_mbar_init();
    tma_prefetch_desc(&maps.q32);
    tma_prefetch_desc(&maps.k32);
    tma_prefetch_desc(&maps.v);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
#ifdef KDA_PROFILE
  if (tid == 0 && (blockIdx.x | blockIdx.y | blockIdx.z) == 0)
    reinterpret_cast<uint64_t*>(p.status)[41] = globaltimer_ns() - kt0;
#endif
  // Shared-memory matrix descriptors, built once: adding (byte offset >> 4) to a
  // descriptor moves its start address (all addresses stay below 256 KB).
  const uint32_t sbase = smem_u32(sm);
  const uint64_t D_SW128 = sdesc_sw128(sbase);                        // K-major, 128-B swizzle
  const uint64_t D_ST = sdesc(sbase + OFF_ST, 8192, 512, 4);          // S, MN-major 64-B swizzle
  const uint64_t D_VNT = sdesc(sbase + OFF_SLOT + S_U, 4096, 512, 4);  // v_new of slot 0, MN-major 64-B swizzle
  auto d128 = [&](uint32_t off) { return D_SW128 + (off >> 4); };
  const size_t state_off = (static_cast<size_t>(seq) * HV + hv) * KD * VD;

  if (warp < NPROD / 32) {
    // ============================== producer ===============================
    uint8_t* pb = sm + OFF_PREP;  // the prep:: tiles
    const int pt = tid;           // 0..255
    const int dp = pt & 63;       // key dims 2 dp, 2 dp + 1 owned in the elementwise pass
    const int hq = pt >> 6;       // ... for rows [16 hq, 16 hq + 16)
    const int quad = warp & 3;    // TMEM lane quadrant of this warp
    const int cpart = warp >> 2;  // which half of a readout this warp takes
    const float scale = p.scale;
    const uint64_t D_PREP = sdesc_sw128(sbase + OFF_PREP);
    const uint64_t D_KD_MN = sdesc(sbase + OFF_PREP + prep::KDT, 8192, 1024, 2);  // kd as MN-major B
    const uint64_t D_V_MN = sdesc(sbase + OFF_PREP + prep::VRAW, 8192, 1024, 2);  // v as MN-major B
    uint32_t pmma_phase = 0, pmma_issued = 0;
    bool raw_pending = false;
    int raw_pending_j = 0;
    bool failed = false, range_bad = false;
    auto timeout = [&]() {
      failed = true;
      atomicOr(p.status, kStatusTimeout);
    };
    PROF_DECL

    auto issue_raw = [&](int m, int j) {  // elected: TMA q, k, v tiles of chunk m (own chunk j)
      prep::issue_raw(pb, &maps.q32, &maps.k32, &maps.v, &bars[B_RAW], hk, hv, static_cast<int>(tok0) + m * C);
      raw_pending = true;
      raw_pending_j = j;
    };
    // g of this thread's 16 rows x 2 dims (and beta) arrive in registers in four
    // 4-row parts issued at different points of the previous chunk, so that few
    // loads are in flight at once
    float2 gpre[16];
    float bpre = 0.f;
    auto prefetch_gb = [&](int m, int part) {
      const int rows = min(C, len - m * C);
      const long base = tok0 + static_cast<long>(m) * C;
      // unconditional loads (rows past the end read the last row; finish_gate_rows masks them)
      if (PRE) {  // raw gate input, bf16 pairs (kept raw in .x)
#pragma unroll
        for (int i = 4 * part; i < 4 * part + 4; ++i) {
          const int c = min(16 * hq + i, rows - 1);
          gpre[i].x = __uint_as_float(
              __ldg(reinterpret_cast<const uint32_t*>(p.g_raw + (static_cast<size_t>(base + c) * HV + hv) * KD) + dp));
        }
      } else {
#pragma unroll
        for (int i = 4 * part; i < 4 * part + 4; ++i) {
          const int c = min(16 * hq + i, rows - 1);
          gpre[i] = __ldg(reinterpret_cast<const float2*>(p.g + (static_cast<size_t>(base + c) * HV + hv) * KD) + dp);
        }
      }
      if (part == 0 && pt < C) bpre = __ldg(p.beta + static_cast<size_t>(base + min(pt, rows - 1)) * HV + hv);
    };
    bool pub_pending = false;  // record j-1 stored but not yet published
    // Record jp is complete in the ring: tell the NSLICE consumers, one lane each
    // (called by a whole warp; lane 0 first waits until record jp - 2, whose
    // publish phase the consumers' barrier must have left, is loaded everywhere).
    // A release arrive at cluster scope costs the issuing thread on the order of a
    // thousand cycles, so the four go out as one warp instruction.
    auto publish = [&](int jp) {
      bool ok = true;
      if (lane == 0) {
        fence_proxy_async_global();
        if (jp >= 2) ok = mbar_wait_cluster(&bars[B_ACK + (jp & 1)], ((jp - 2) >> 1) & 1, p.wait_ns);
        if (!ok) timeout();
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (ok && lane < NSLICE)
        mbar_arrive_cluster(mapa_shared(smem_u32(&bars[B_PUB + 2 * rank + (jp & 1)]), static_cast<uint32_t>(lane)));
      __syncwarp();
    };

    const int first = static_cast<int>(rank);
    if (first < NT) {
      if (pt == 0) issue_raw(first, 0);
#pragma unroll
      for (int part = 0; part < 4; ++part) prefetch_gb(first, part);
    }
    int j = 0;
    for (int m = first; m < NT; m += NSLICE, ++j) {
      uint8_t* gs = ring + static_cast<size_t>(m % RING) * GSLOT;
      const int rows = min(C, len - m * C);
      const bool next = m + NSLICE < NT;
      // ---- 1. raw q, k, v of chunk m (and the gate parameters of the pre-stage) ----
      float a_log = 0.f;
      float2 dt = make_float2(0.f, 0.f);
      if (PRE) {
        a_log = __ldg(p.A_log + hv);
        dt = __ldg(reinterpret_cast<const float2*>(p.dt_bias + static_cast<size_t>(hv) * KD) + dp);
      }
      if (!mbar_wait(&bars[B_RAW], j & 1, p.wait_ns)) timeout();
      if (pt == 0) bulk_wait_read();  // the previous record's Aqk, W and U stagings have been read
      prep::finish_gate_rows<PRE>(gpre, bpre, hq, pt, rows);
      if (PRE) {  // activations, and the raw q, k row norms (read before the pass rewrites the rows)
        prep::activate(gpre, bpre, p.prestage, p.lower_bound, expf(a_log), dt, hq, pt, rows);
        prep::row_norms(pb, rn, pt);
      }
      if (pt < C) beta_s[pt] = bpre;
      {
        float2 qsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          qsum.x += gpre[i].x;
          qsum.y += gpre[i].y;
        }
        reinterpret_cast<float2*>(gsum + hq * KD)[dp] = qsum;
      }
      if (role_any(NB_PREP, NPROD, failed)) break;
      if (pt == 0) raw_pending = false;
      PROF(0);

      // ---- 2. elementwise: operand tiles; qd, kr^T and e^{g_last} straight into the
      //         record (a slot is rewritten only after its previous record was loaded
      //         everywhere: publish() of the record two before waited for that) ----
      {
        if (PRE)
          prep::elementwise<false, true>(pb, gsum, gpre, dp, hq, rows, scale, gs + R_WQ + R_QD_IN_KB, R_W_KB,
                                         gs + R_KRT, reinterpret_cast<float*>(gs + G_GAM), rn, range_bad);
        else
          prep::elementwise<false, false>(pb, gsum, gpre, dp, hq, rows, scale, gs + R_WQ + R_QD_IN_KB, R_W_KB,
                                          gs + R_KRT, reinterpret_cast<float*>(gs + G_GAM), nullptr, range_bad);
      }
      fence_proxy_async_global();  // the record's plain stores, read by the chains' bulk copies
      if (pt == 0 && pub_pending) bulk_wait_group<0>();  // the previous record's W/U stores have landed
      fence_proxy_async_smem();
      role_sync(NB_PREP, NPROD);
      PROF(1);
      // The previous record goes out from warp 3 while warp 0 issues the MMAs below
      // (the cluster-scope arrives cost the issuing warp about a thousand cycles, and
      // would also wait for its g loads, so it publishes before requesting them).
      // Thread 0's wait on the record's stores is ordered before this by the barrier.
      if (pub_pending) {
        if (warp == 3) publish(j - 1);
        pub_pending = false;
      }

      // ---- 3. the diagonal halves and the block below them of L and Aqk ----
      if (warp == 0) {
        tc_fence_after();
        prep::issue_lqk(tmem, D_PREP);
        umma_commit_warp(&bars[B_PMMA]);
        ++pmma_issued;
      }
      if (next) prefetch_gb(m + NSLICE, 0);
      __syncwarp();
      if (mbar_wait(&bars[B_PMMA], pmma_phase & 1, p.wait_ns)) ++pmma_phase;  // else still in flight: drained below
      else timeout();
      tc_fence_after();
      PROF(2);

      // ---- 4. TMEM -> M (fp32), Aqk ----
      prep::readout_lqk(pb, tmem, beta_s, quad, cpart, lane);
      tc_fence_before();
      fence_proxy_async_smem();
      if (role_any(NB_PREP, NPROD, failed)) break;
      if (pt == 0) {
        bulk_store(gs + R_AQK, pb + prep::AQK_STG, 8192);
        bulk_commit();
      }
      if (next) prefetch_gb(m + NSLICE, 1);
      PROF(3);

      // ---- 5. T = (I + M)^{-1} and A = T Diag(beta): diagonal blocks, then the block columns ----
      prep::inverse_diag_blocks(pb, beta_s, warp, pt, lane);
      role_sync(NB_PREP, NPROD);
      PROF(4);
      // next chunk's g: requested here, so the loads are in flight during the
      // inverse rather than in front of the barrier below
      if (next) prefetch_gb(m + NSLICE, 2);
      PROF(10);
      if (warp < 3)
        inverse_block_columns(reinterpret_cast<float*>(pb + prep::MB), beta_s, pb + prep::AMAT, warp, lane);
      PROF(5);
      if (pt == 0) bulk_wait_read();  // the Aqk staging has been read: its buffer takes U next
      fence_proxy_async_smem();
      role_sync(NB_PREP, NPROD);
      PROF(6);

      // ---- 6. W = A kd, U = A v (kd and v as MN-major B operands) ----
      if (pt == 0) {
        if (!failed) {
          tc_fence_after();
          constexpr uint32_t idesc = idesc_f16kind(64, 128) | IDESC_B_MN_MAJOR;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ad = D_PREP + ((prep::AMAT + ks * 32) >> 4);
            umma_f16(tmem + TM_W, ad, D_KD_MN + ((ks * 2048) >> 4), idesc, ks != 0);
            umma_f16(tmem + TM_U, ad, D_V_MN + ((ks * 2048) >> 4), idesc, ks != 0);
          }
          umma_commit(&bars[B_PMMA]);
          ++pmma_issued;
        }
      }
      if (next) prefetch_gb(m + NSLICE, 3);
      __syncwarp();
      if (mbar_wait(&bars[B_PMMA], pmma_phase & 1, p.wait_ns)) ++pmma_phase;  // else still in flight: drained below
      else timeout();
      tc_fence_after();
      // the stacked tile (M and A by now) and v are free again: fetch the next own chunk
      if (pt == 0 && next && !failed) issue_raw(m + NSLICE, j + 1);
      PROF(7);

      // ---- 7. W -> staging over kd (bf16 SW128), U -> staging over cA (4 slices of [64 x 32] bf16) ----
      __syncwarp();
      {
        const int i = 16 * quad + (lane & 15);
        const uint32_t tcol = cpart == 0 ? TM_W : TM_U;
#pragma unroll
        for (int q2 = 0; q2 < 4; q2 += 2) {
          float r0[32], r1[32];
          tmem_ld32(tmem_addr(tmem, 32 * quad, tcol + 32 * q2), r0);
          tmem_ld32(tmem_addr(tmem, 32 * quad, tcol + 32 * (q2 + 1)), r1);
          tmem_ld_wait();
          if (lane < 16) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float* r = h ? r1 : r0;
              const int q4 = q2 + h;
#pragma unroll
              for (int j8 = 0; j8 < 4; ++j8) {
                uint8_t* d8 = cpart == 0 ? pb + prep::KDT + sw128_offset(i, 32 * q4 + 8 * j8, 64)
                                         : pb + prep::USTG + q4 * 4096 + i * (VS * 2) + 16 * j8;
                st_v4(d8, pack2(r[8 * j8], r[8 * j8 + 1]), pack2(r[8 * j8 + 2], r[8 * j8 + 3]),
                      pack2(r[8 * j8 + 4], r[8 * j8 + 5]), pack2(r[8 * j8 + 6], r[8 * j8 + 7]));
              }
            }
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      if (role_any(NB_PREP, NPROD, failed)) break;
      PROF(8);

      // ---- 8. W/U to the ring; the record is published early in the next chunk
      //         (or at the end), once these stores have landed.  The first record
      //         goes out at once: every chain of the cluster is waiting for it. ----
      if (pt == 0) {
        bulk_store(gs + R_WQ, pb + prep::KDT, 8192);
        bulk_store(gs + R_WQ + R_W_KB, pb + prep::KDT + 8192, 8192);
        bulk_store(gs + G_U, pb + prep::USTG, 16384);
        bulk_commit();
        if (j == 0) bulk_wait_group<0>();
      }
      pub_pending = true;
      if (j == 0) {
        role_sync(NB_PREP, NPROD);
        if (warp == 3) publish(0);
        pub_pending = false;
      }
      PROF(9);
    }
    if (range_bad) atomicOr(p.status, kStatusRange);
    if (warp == 0 && pub_pending) {  // the last record (warp-uniform decision)
      if (!__any_sync(0xFFFFFFFFu, failed)) {
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        publish(j - 1);
      }
      pub_pending = false;
    }
    // drain after an abort: copies and MMAs this role issued must finish first
    if (pt == 0) {
      if (raw_pending && !mbar_wait(&bars[B_RAW], raw_pending_j & 1, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
      if (pmma_issued > pmma_phase && !mbar_wait(&bars[B_PMMA], (pmma_issued - 1) & 1, DRAIN_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
      bulk_wait_all();
      // records this CTA published must be loaded everywhere before it exits
      for (int jj = (j >= 2 ? j - 2 : 0); !failed && jj < j; ++jj)
        if (!mbar_wait_cluster(&bars[B_ACK + (jj & 1)], (jj >> 1) & 1, p.wait_ns))
          atomicOr(p.status, kStatusTimeout);
      PROF_STORE(0);
    }
    __syncwarp();
  } else {
    // ================================ chain ================================
    const int qt = tid - NPROD;  // state row d
    const int qw = warp & 3;     // TMEM lane quadrant
    const int d = qt;
    float st[VS];
    if (p.s0) {
      const float4* src = reinterpret_cast<const float4*>(p.s0 + state_off + static_cast<size_t>(d) * VD + v0);
#pragma unroll
      for (int j4 = 0; j4 < VS / 4; ++j4) {
        const float4 v4 = src[j4];
        st[4 * j4] = v4.x;
        st[4 * j4 + 1] = v4.y;
        st[4 * j4 + 2] = v4.z;
        st[4 * j4 + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < VS; ++jj) st[jj] = 0.f;
    }
    auto write_st = [&]() {  // row d of S as bf16, MN-major 64-byte swizzle
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        st_v4(sm + OFF_ST + mn_sw64_offset(d, 8 * ch), pack2(st[8 * ch], st[8 * ch + 1]),
              pack2(st[8 * ch + 2], st[8 * ch + 3]), pack2(st[8 * ch + 4], st[8 * ch + 5]),
              pack2(st[8 * ch + 6], st[8 * ch + 7]));
    };
    write_st();
    fence_proxy_async_smem();
    role_sync(NB_CHAIN, NCHAIN);

    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    bool failed = false, aborted = false;
    int a_issued = 0, b_issued = 0, c_issued = 0, a_done = 0, b_done = 0, c_done = 0;
    auto timeout = [&]() {
      failed = true;
      atomicOr(p.status, kStatusTimeout);
    };
    // Record loads (thread kLoader, in a warp that only emits o rows while the state
    // product runs): chunk m goes to slot m & 1 once it is published by producer
    // m % 4 (its record j = m / 4) and the slot is free.
    constexpr int kLoader = 64;
    constexpr int kIssuer = 96;  // MMA issue (warp 11, lane 0)
    int next_load = 0;       // first chunk whose load is not issued yet
    int loads_done = 0;      // loads whose FULL phase was observed (and acknowledged)
    auto pub_bar = [&](int m) { return &bars[B_PUB + 2 * (m % NSLICE) + ((m / NSLICE) & 1)]; };
    auto issue_load = [&](int m) {
      fence_proxy_async_global();
      const int s = m & 1;
      uint8_t* slot = sm + OFF_SLOT + s * SSLOT;
      const uint8_t* gs = ring + static_cast<size_t>(m % RING) * GSLOT;
      mbar_arrive_expect_tx(&bars[B_FULL + s], REC_TX);
      bulk_load(slot + R_WQ, gs + R_WQ, R_TILES, &bars[B_FULL + s]);
      bulk_load(slot + S_U, gs + G_U + rank * 4096, 4096, &bars[B_FULL + s]);
      bulk_load(slot + S_GAM, gs + G_GAM, 512, &bars[B_FULL + s]);
    };
    // Issue the loads of chunks below `limit` that are published (chunk `need`, if
    // not yet issued, is waited for).  Chunk m + 1 goes to the slot of chunk m - 1,
    // so it is only issued once chunk m - 1's last MMA (B_C) has completed.
    auto pump_loads = [&](int limit, int need) {
      while (next_load < NT && next_load < limit) {
        const int m = next_load;
        if (!mbar_try_wait_cluster(pub_bar(m), (m / NSLICE >> 1) & 1)) {
          if (m != need) return;
          if (!mbar_wait_cluster(pub_bar(m), (m / NSLICE >> 1) & 1, p.wait_ns)) {
            timeout();
            return;
          }
        }
        issue_load(m);
        ++next_load;
      }
    };
    // o rows of chunk m: lanes 64-127 of D_A[m & 1] (rewritten only by chunk m + 2's MMAs),
    // read by the two warps of lane quadrants 2 and 3
    auto emit_o = [&](int m) {
      const int rows = min(C, len - m * C);
      if (qw < 2) return;  // only the warps of lane quadrants 2 and 3 read o
      if (mbar_wait(&bars[B_C], m & 1, p.wait_ns)) ++c_done;  // else drained below
      else timeout();
      if (p.h) return;  // state pass: no output
      __syncwarp();
      tc_fence_after();
      float orr[32];
      tmem_ld32(tmem_addr(tmem, 32 * qw, TM_A0 + 32 * (m & 1)), orr);
      tmem_ld_wait();
      const int c = 32 * (qw - 2) + lane;
      if (c < rows) {
        uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(tok0 + m * C + c) * HV + hv) * VD + v0);
#pragma unroll
        for (int j8 = 0; j8 < VS / 8; ++j8)
          dst[j8] = make_uint4(pack2(orr[8 * j8], orr[8 * j8 + 1]), pack2(orr[8 * j8 + 2], orr[8 * j8 + 3]),
                               pack2(orr[8 * j8 + 4], orr[8 * j8 + 5]), pack2(orr[8 * j8 + 6], orr[8 * j8 + 7]));
      }
    };
    // All chain MMAs are issued by one lane of a warp that otherwise only emits o rows,
    // so the warps that compute v_new and the state never wait on an issue.  The
    // o-side product of chunk m (Aqk v_new) is issued after chunk m + 1's state
    // product, when it no longer delays anything on the recurrence.
    auto issue_o_update = [&](int mc) {  // issuer: o rows of chunk mc += Aqk v_new
      const int sc = mc & 1;
      const uint32_t soc = OFF_SLOT + sc * SSLOT;
      constexpr uint32_t idesc = idesc_f16kind(128, VS) | IDESC_B_MN_MAJOR;
      // the 128 rows starting 64 rows before Aqk (kr^T rows 64..127, then Aqk): Aqk v_new
      // lands in lanes 64-127 next to qd S; lanes 0-63 (X, consumed) take a harmless product
      if (!p.h)  // (the state pass keeps the commit, so the barrier's phases stay in step)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16(tmem + TM_A0 + 32 * sc, d128(soc + R_AQK - 8192 + ks * 32),
                   D_VNT + ((sc * SSLOT + ks * 1024) >> 4), idesc, 1u);
      umma_commit(&bars[B_C]);
      ++c_issued;
    };
    PROF_DECL
    if (qt == kLoader) pump_loads(2, -1);
    for (int m = 0; m < NT; ++m) {
      const int s = m & 1;
      const uint32_t so = OFF_SLOT + s * SSLOT;  // this chunk's record slot
      uint8_t* slot = sm + so;
      if (p.h) {  // state pass: row d, columns v0 .. v0 + 31 of the state entering chunk m
        uint4* dst = reinterpret_cast<uint4*>(
            p.h + ((static_cast<size_t>(seq) * HV + hv) * p.h_chunks + m) * KD * VD + static_cast<size_t>(d) * VD + v0);
#pragma unroll
        for (int j8 = 0; j8 < VS / 8; ++j8)
          dst[j8] = make_uint4(pack2(st[8 * j8], st[8 * j8 + 1]), pack2(st[8 * j8 + 2], st[8 * j8 + 3]),
                               pack2(st[8 * j8 + 4], st[8 * j8 + 5]), pack2(st[8 * j8 + 6], st[8 * j8 + 7]));
      }
      if (qt == kLoader && !failed) pump_loads(m + 1, m);
      PROF(6);
      __syncwarp();
      if (!mbar_wait(&bars[B_FULL + s], (m >> 1) & 1, p.wait_ns)) timeout();
      if (qt == kLoader && !failed) ++loads_done;
      PROF(0);
      // ---- [X ; O] = [W ; qd] S (one M = 128 accumulator), then chunk m - 1's o update ----
      if (qt == kIssuer && !failed) {
        // Record m is in shared memory (its bulk loads have completed): release its
        // ring slot.  Nothing of the slot is read after this, so the arrive needs no
        // ordering of its own.
        mbar_arrive_cluster_relaxed(
            mapa_shared(smem_u32(&bars[B_ACK + ((m / NSLICE) & 1)]), static_cast<uint32_t>(m % NSLICE)));
        tc_fence_after();
        constexpr uint32_t idesc = idesc_f16kind(128, VS) | IDESC_B_MN_MAJOR;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_f16(tmem + TM_A0 + 32 * s, d128(so + R_WQ + kb * R_W_KB + ks * 32),
                     D_ST + (((kb * 4 + ks) * 1024) >> 4), idesc, (kb | ks) != 0);
        umma_commit(&bars[B_A]);
        ++a_issued;
        if (m > 0) issue_o_update(m - 1);
      }
      __syncwarp();
      if (m > 0) emit_o(m - 1);  // previous chunk's rows, while this chunk's MMAs run
      // chunk m - 1 is finished with its slot (its reads ended before the last
      // barrier of that chunk, its last MMA with emit_o): chunk m + 1 may load
      if (qt == kLoader && !failed) pump_loads(m + 2, -1);
      if (mbar_wait(&bars[B_A], m & 1, p.wait_ns)) ++a_done;  // else drained below
      else timeout();
      __syncwarp();
      tc_fence_after();
      PROF(1);
      // ---- v_new = U - X  ->  bf16 MN-major over the U rows (row c = token; lane
      //      quadrants 0 and 1; each thread rewrites the 64 bytes of its own row) ----
      if (qw < 2) {
        float xr[32];
        tmem_ld32(tmem_addr(tmem, 32 * qw, TM_A0 + 32 * s), xr);
        const int c = 32 * qw + lane;
        uint8_t* urow = slot + S_U + c * (VS * 2);
        uint4 u[4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) u[ch] = reinterpret_cast<const uint4*>(urow)[ch];
        tmem_ld_wait();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t uw[4] = {u[ch].x, u[ch].y, u[ch].z, u[ch].w};
          uint32_t w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float lo = __uint_as_float(uw[t] << 16) - xr[8 * ch + 2 * t];
            const float hi = __uint_as_float(uw[t] & 0xFFFF0000u) - xr[8 * ch + 2 * t + 1];
            w[t] = pack2(lo, hi);
          }
          st_v4(slot + S_U + mn_sw64_offset(c, 8 * ch), w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (role_any(NB_CHAIN, NCHAIN, failed)) {
        aborted = true;
        break;
      }
      PROF(2);
      // ---- P = kr^T v_new ----
      if (qt == kIssuer) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_f16kind(128, VS) | IDESC_B_MN_MAJOR;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16(tmem + TM_P, d128(so + R_KRT + ks * 32), D_VNT + ((s * SSLOT + ks * 1024) >> 4), idesc, ks != 0);
        umma_commit(&bars[B_B]);
        ++b_issued;
      }
      __syncwarp();
      if (mbar_wait(&bars[B_B], m & 1, p.wait_ns)) ++b_done;  // else drained below
      else timeout();
      __syncwarp();
      tc_fence_after();
      PROF(3);
      // ---- S <- Diag(e^{g_last}) S + P ; refresh the bf16 copy ----
      {
        float pr[32];
        tmem_ld32(tmem_addr(tmem, 32 * qw, TM_P), pr);
        const float gmm = reinterpret_cast<const float*>(slot + S_GAM)[d];
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < VS; ++jj) st[jj] = fmaf(gmm, st[jj], pr[jj]);
        write_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (role_any(NB_CHAIN, NCHAIN, failed)) {
        aborted = true;
        break;
      }
      PROF(4);
    }
    if (!aborted && !failed && NT > 0 && qt == kIssuer) {
      tc_fence_after();
      issue_o_update(NT - 1);
    }
#ifdef KDA_PROFILE
    if (qt == 0 && (blockIdx.x | blockIdx.y | blockIdx.z) == 0)
      reinterpret_cast<uint64_t*>(p.status)[42] = globaltimer_ns() - kt0;
#endif
    if (!aborted && !failed && NT > 0) {
      __syncwarp();
      emit_o(NT - 1);
    }
    if (qt == kIssuer) {  // drain MMAs still in flight after an abort
      if (a_issued > a_done && !mbar_wait(&bars[B_A], (a_issued - 1) & 1, DRAIN_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
      if (b_issued > b_done && !mbar_wait(&bars[B_B], (b_issued - 1) & 1, DRAIN_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
      if (c_issued > c_done && !mbar_wait(&bars[B_C], (c_issued - 1) & 1, DRAIN_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
    }
    if (qt == 0) PROF_STORE(16);
    if (qt == kLoader)  // record loads still in flight after an abort
      for (int m = loads_done; m < next_load; ++m)
        if (!mbar_wait(&bars[B_FULL + (m & 1)], (m >> 1) & 1, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
    __syncwarp();
    if (p.sfin && !aborted && !failed) {
      float4* dst = reinterpret_cast<float4*>(p.sfin + state_off + static_cast<size_t>(d) * VD + v0);
#pragma unroll
      for (int j4 = 0; j4 < VS / 4; ++j4)
        dst[j4] = make_float4(st[4 * j4], st[4 * j4 + 1], st[4 * j4 + 2], st[4 * j4 + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
#ifdef KDA_PROFILE
  if (tid == 0 && (blockIdx.x | blockIdx.y | blockIdx.z) == 0)
    reinterpret_cast<uint64_t*>(p.status)[43] = globaltimer_ns() - kt0;
#endif
  cluster_sync_all();  // no CTA leaves while a peer may still arrive on its barriers
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
#ifdef KDA_PROFILE
  if (tid == 0 && rank == 0 && blockIdx.y + gridDim.y * blockIdx.z < 32) {
    const int c = blockIdx.y + gridDim.y * blockIdx.z;
    reinterpret_cast<uint64_t*>(p.status)[64 + 2 * c] = kt0;
    reinterpret_cast<uint64_t*>(p.status)[65 + 2 * c] = globaltimer_ns();
  }
#endif
}

// ======================================================================
// Split chunk kernel: the roles of the cluster kernel above on separate SMs.
// One cooperative launch over every SM: CTA b < NU is the chain of unit b (one
// (sequence, value head) with the whole K x V state, 16 warps); every other
// CTA runs two independent 8-warp producer pipelines.  Records are produced in
// chunk-major order over all units, written to the per-unit L2 ring and
// announced with a GPU-scope ready flag; the chain raises a per-unit counter of
// loaded chunks, which bounds how far producers may run ahead of it (a ring
// slot is rewritten only after its previous record was loaded).  All CTAs are
// resident at once (cooperative launch), and every wait is bounded.
// ======================================================================
namespace split {
constexpr int NTHREADS = 512;
// ring slots a unit's producers may fill ahead of its chain (of the RING slots the
// workspace holds): few enough that a record is still in L2 when the chain loads it
#ifndef SPLIT_RING
#define SPLIT_RING 16
#endif
constexpr int SRING = SPLIT_RING;
static_assert(SRING >= 2 && SRING <= RING, "split ring depth");
constexpr uint32_t PIPE = 256;              // threads of one producer pipeline
// Record of one chunk as the split kernel lays it out in a ring slot (bf16 tiles in the
// 128-byte swizzle layout, each the byte image of a tcgen05 B operand).  Part A is
// what the chain needs first and is copied on its own.
constexpr uint32_t SR_QW = 0;                 // 2 K-blocks (16 KB apart) x [qd rows | W rows]
constexpr uint32_t SR_KB = 16384;
constexpr uint32_t SR_W_IN_KB = 8192;
constexpr uint32_t SR_GAM = 32768;            // e^{g_last} [128] fp32
constexpr uint32_t REC_A_BYTES = SR_GAM + 512;
constexpr uint32_t SR_KRT = 33792;            // kr^T [128 x 64], then Aqk [64 x 64]: one 192-row operand
constexpr uint32_t SR_AQK = SR_KRT + 16384;
constexpr uint32_t SR_U = SR_AQK + 8192;      // U^T [128 x 64] (rows = value columns)
constexpr uint32_t REC_BYTES = SR_U + 16384;  // 74,752 B
static_assert(REC_BYTES <= GSLOT, "record fits a ring slot");
// producer pipeline region (offsets from the region base, 1024-aligned): the prep:: tiles,
// then beta, the quarter sums of g, barriers and the ring-slot flag
constexpr uint32_t P_BETA = prep::QDS + 16384, P_GSUM = P_BETA + 256, P_RN = P_GSUM + 2048, P_BAR = P_RN + 512,
                   P_STRIDE = 109568;
static_assert(P_BAR + 64 <= P_STRIDE && P_STRIDE % 1024 == 0, "producer pipeline region");
// chain region
// chain region: record part A ([qd; W], e^{g_last}) in three buffers, part B (kr^T, Aqk,
// U^T) in two, then the o staging tiles
constexpr uint32_t PA_STRIDE = 33792;          // REC_A_BYTES rounded up to 1 KB
constexpr uint32_t PB_STRIDE = REC_BYTES - SR_KRT;
constexpr uint32_t C_PA = 0;
constexpr uint32_t C_PB = C_PA + 3 * PA_STRIDE;
constexpr uint32_t C_STG = C_PB + 2 * PB_STRIDE;  // two 16 KB o staging tiles ([token][v], two 64-column halves)
constexpr uint32_t C_BAR = C_STG + 2 * 16384;
constexpr uint32_t C_MISC = C_BAR + 128;       // tmem base
// the TMEM base address lives past both roles' regions (chain profile stamps at C_MISC + 64)
constexpr uint32_t TMEM_SLOT = (2 * P_STRIDE > C_MISC + 448 ? 2 * P_STRIDE : C_MISC + 448);
constexpr uint32_t SMEM_BYTES = TMEM_SLOT + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;
static_assert(SMEM_ALLOC <= 232448, "split kernel shared memory");
static_assert(PA_STRIDE >= REC_A_BYTES && PA_STRIDE % 1024 == 0 && PB_STRIDE % 1024 == 0 && C_PB % 1024 == 0,
              "record buffers keep the 1 KB alignment of the swizzled operands");
constexpr int CB_FULL = 0, CB_B = 3;  // chain barriers (CB_FULL: [3], one per part-A buffer)
constexpr int PB_RAW = 0, PB_PMMA = 1;                     // producer barriers (per pipeline)
constexpr uint32_t P_SLOT_FREE = P_BAR + 32;               // shared flag: the record's ring slot may be written
constexpr uint32_t NB_CHAIN_ALL = 3;

struct Rec {
  int m, u, seq, hv, hk, len;
  long tok0;
};
// Record r of the chunk-major enumeration: chunk r / NU of the launch's unit r % NU (x.u,
// which indexes the ring and the flags; the unit of the problem is p.unit0 + x.u); false
// when the unit has no such chunk.
__device__ __forceinline__ bool rec_at(const FwdParams& p, int NU, int r, Rec& x) {
  x.m = r / NU;
  x.u = r - x.m * NU;
  const int ug = p.unit0 + x.u;
  x.seq = ug / p.HV;
  x.hv = ug - x.seq * p.HV;
  x.hk = x.hv / (p.HV / p.H);
  seq_range(p, x.seq, x.tok0, x.len);
  return x.m * C < x.len;
}
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* a, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
// element (k, n) of an MN-major 128-byte-swizzled bf16 operand whose N = 128 columns
// form two 64-column atoms `atom_stride` bytes apart (8-row K groups 1024 B apart)
__device__ __forceinline__ uint32_t mn_sw128_offset(uint32_t k, uint32_t n, uint32_t atom_stride) {
  return (n >> 6) * atom_stride + (k >> 3) * 1024u + (k & 7u) * 128u + (((((n & 63u) >> 3) ^ (k & 7u))) << 4) +
         (n & 7u) * 2u;
}

// ------------------------------------------------------------ producer ----
constexpr int kRecStorer = 32;  // pipeline thread storing qd and kr^T to the ring (warp 1)
// -DKDA_PROFILE: clock64 stamps of thread 0 of pipeline 0 at numbered points of its
// record KDA_STAMP_RECORD, written straight to the workspace words [480, 498) (below the
// record flags at byte kFlagOffset)
#ifndef KDA_STAMP_RECORD
#define KDA_STAMP_RECORD 4
#endif
#ifndef KDA_STAMP_M0  // first of the 64 chunks of unit 0 whose publication and copies are stamped
#define KDA_STAMP_M0 0
#endif
#ifdef KDA_PROFILE
#define PSTAMP(i)                                                                     \
  do {                                                                                \
    if (q == 0 && j == KDA_STAMP_RECORD && pt == 0) {                                 \
      long long t_;                                                                   \
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(t_)::"memory");                    \
      reinterpret_cast<volatile long long*>(p.status)[480 + (i)] = t_;                \
    }                                                                                 \
  } while (0)
#else
#define PSTAMP(i) \
  do {            \
  } while (0)
#endif
template <bool PRE>
__device__ __forceinline__ void producer(const Maps& maps, const FwdParams& p, uint8_t* sm, uint32_t tmem,
                                         int pipe, int q, int NQ, int NU, int NREC_BOUND, uint32_t* flags) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pt = tid & 255;
  const int pw = warp & 7;       // warp within the pipeline
  const int dp = pt & 63;        // key dims 2 dp, 2 dp + 1 in the elementwise pass
  const int hq = pt >> 6;        // ... rows [16 hq, 16 hq + 16)
  const int quad = warp & 3;     // TMEM lane quadrant
  const int cpart = pw >> 2;     // half of a readout
  const uint32_t NB = 1 + static_cast<uint32_t>(pipe);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + P_BAR);
  float* beta_s = reinterpret_cast<float*>(sm + P_BETA);
  float* gsum = reinterpret_cast<float*>(sm + P_GSUM);
  float* rnorm = reinterpret_cast<float*>(sm + P_RN);  // row norms of the raw q, k (pre-stage)
  volatile uint32_t* slot_free = reinterpret_cast<volatile uint32_t*>(sm + P_SLOT_FREE);
  const uint32_t sb = smem_u32(sm);
  const uint64_t D_PREP = sdesc_sw128(sb);
  const uint64_t D_KD_MN = sdesc(sb + prep::KDT, 8192, 1024, 2);
  const uint64_t D_V_MN = sdesc(sb + prep::VRAW, 8192, 1024, 2);
  const int HV = p.HV;
  const float scale = p.scale;
  uint32_t pmma_phase = 0, pmma_issued = 0;
  bool raw_pending = false;
  int raw_pending_j = 0;
  bool failed = false, range_bad = false;
  auto timeout = [&]() {
    failed = true;
    atomicOr(p.status, kStatusTimeout);
#ifdef KDA_PROFILE
    atomicCAS(reinterpret_cast<unsigned long long*>(p.status) + 400, 0ull,
              (static_cast<unsigned long long>(blockIdx.x) << 40) | (static_cast<unsigned long long>(threadIdx.x) << 24) | 20ull);
#endif
  };
  auto issue_raw = [&](const Rec& x, int jj) {  // elected
    prep::issue_raw(sm, &maps.q32, &maps.k32, &maps.v, &bars[PB_RAW], x.hk, x.hv, static_cast<int>(x.tok0) + x.m * C);
    raw_pending = true;
    raw_pending_j = jj;
  };
  float2 gpre[16];
  float bpre = 0.f;
  auto prefetch_gb = [&](const Rec& x, int part) {
    const int rows = min(C, x.len - x.m * C);
    const long base = x.tok0 + static_cast<long>(x.m) * C;
    // unconditional loads (rows past the end read the last row; finish_gate_rows masks them)
    if (PRE) {  // raw gate input, bf16 pairs (kept raw in .x)
#pragma unroll
      for (int i = 4 * part; i < 4 * part + 4; ++i) {
        const int c = min(16 * hq + i, rows - 1);
        gpre[i].x = __uint_as_float(
            __ldg(reinterpret_cast<const uint32_t*>(p.g_raw + (static_cast<size_t>(base + c) * HV + x.hv) * KD) + dp));
      }
    } else {
#pragma unroll
      for (int i = 4 * part; i < 4 * part + 4; ++i) {
        const int c = min(16 * hq + i, rows - 1);
        gpre[i] = __ldg(reinterpret_cast<const float2*>(p.g + (static_cast<size_t>(base + c) * HV + x.hv) * KD) + dp);
      }
    }
    if (part == 0 && pt < C) bpre = __ldg(p.beta + static_cast<size_t>(base + min(pt, rows - 1)) * HV + x.hv);
  };

  // Records of this launch: chunk-major over its units, up to the longest of their
  // sequences (the host passes a bound; with cu_seqlens the lengths are read here, so
  // that no pipeline walks the empty tail of a bound set by the packed total)
  int NREC = NREC_BOUND;
  if (p.cu) {
    int mx = 0;
    for (int sq = p.unit0 / HV; sq <= (p.unit0 + NU - 1) / HV; ++sq) {
      long t0;
      int len;
      seq_range(p, sq, t0, len);
      mx = max(mx, (len + C - 1) / C);
    }
    NREC = min(NREC_BOUND, mx * NU);
  }
  auto next_valid = [&](int r, Rec& x) {
    while (r < NREC && !rec_at(p, NU, r, x)) r += NQ;
    return r;
  };
  // announce record (m, u): its tiles and e^{g_last} are in the ring (called by one
  // thread after a barrier that follows the stores' completion and the writers' fences)
  auto publish = [&](int m, int u) {
    fence_proxy_async_global();
    st_release_gpu(flags + u * 32 + (m % SRING), static_cast<uint32_t>(m + 1));
#ifdef KDA_PROFILE
    if (u == 0 && m >= KDA_STAMP_M0 && m < KDA_STAMP_M0 + 64)
      reinterpret_cast<uint64_t*>(p.status)[200 + m - KDA_STAMP_M0] = globaltimer_ns();
#endif
  };

  Rec cur, nx;
  int r = next_valid(q, cur);
#ifdef KDA_PROFILE
  // [116] the first pipeline found its first record, [117] issued its raw tiles, [118] its gate loads
  if (q == 0 && pt == 0) reinterpret_cast<uint64_t*>(p.status)[116] = globaltimer_ns();
#endif
  if (r < NREC) {
    if (pt == 0) issue_raw(cur, 0);
#ifdef KDA_PROFILE
    if (q == 0 && pt == 0) reinterpret_cast<uint64_t*>(p.status)[117] = globaltimer_ns();
#endif
#pragma unroll
    for (int part = 0; part < 4; ++part) prefetch_gb(cur, part);
#ifdef KDA_PROFILE
    if (q == 0 && pt == 0) reinterpret_cast<uint64_t*>(p.status)[118] = globaltimer_ns();
#endif
  }
  bool pub_pending = false;
  int pub_m = 0, pub_u = 0;
  uint32_t flow_seen = 0u;  // consumed-chunk counter of record flow_n's unit, read ahead
  int flow_n = -1;
  int j = 0;
  for (; r < NREC; ++j) {
    const int rn = next_valid(r + NQ, nx);
    const bool next = rn < NREC;
    uint8_t* gs = p.ring + (static_cast<size_t>(cur.u) * RING + (cur.m % SRING)) * GSLOT;
    const int rows = min(C, cur.len - cur.m * C);
    // ---- 1. raw q, k, v tiles; is the ring slot known to be free (its previous record
    //         loaded by the chain, as the counter read ahead shows)? ----
    float a_log = 0.f;  // gate parameters of the pre-stage, requested before the wait
    float2 dt = make_float2(0.f, 0.f);
    if (PRE) {
      a_log = __ldg(p.A_log + cur.hv);
      dt = __ldg(reinterpret_cast<const float2*>(p.dt_bias + static_cast<size_t>(cur.hv) * KD) + dp);
    }
    PSTAMP(0);
#ifdef KDA_PROFILE
    // [125] the first producer pipeline's first record: loop top, [126] its raw tiles landed
    if (q == 0 && j == 0 && pt == 0) reinterpret_cast<uint64_t*>(p.status)[125] = globaltimer_ns();
#endif
    if (!mbar_wait(&bars[PB_RAW], j & 1, p.wait_ns)) timeout();
#ifdef KDA_PROFILE
    if (q == 0 && j == 0 && pt == 0) reinterpret_cast<uint64_t*>(p.status)[126] = globaltimer_ns();
#endif
    PSTAMP(1);
    if (pt == 0 || pt == kRecStorer) bulk_wait_read();  // the previous record's stagings have been read
    prep::finish_gate_rows<PRE>(gpre, bpre, hq, pt, rows);
    if (PRE) {  // activations, and the raw q, k row norms (read before the pass rewrites the rows)
      prep::activate(gpre, bpre, p.prestage, p.lower_bound, expf(a_log), dt, hq, pt, rows);
      prep::row_norms(sm, rnorm, pt);
    }
    if (pt < C) beta_s[pt] = bpre;
    {
      float2 qsum = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        qsum.x += gpre[i].x;
        qsum.y += gpre[i].y;
      }
      reinterpret_cast<float2*>(gsum + hq * KD)[dp] = qsum;
    }
    const uint32_t need = static_cast<uint32_t>(cur.m - SRING + 1);
    if (pt == kRecStorer) *slot_free = (cur.m < SRING || (flow_n == r && flow_seen >= need)) ? 1u : 0u;
    if (role_any(NB, PIPE, failed)) break;
    PSTAMP(2);
    if (pt == 0) raw_pending = false;
    if (*slot_free == 0u) {
      // Not known: publish this pipeline's previous record first (a chain may be waiting
      // for it, and the ring must never hold a record behind a wait on the chains), then
      // wait for the slot.
      if ((pt == 0 || pt == kRecStorer) && pub_pending) bulk_wait_group<0>();
      role_sync(NB, PIPE);
      if (pub_pending) {
        if (pw == 3 && lane == 0) publish(pub_m, pub_u);
        pub_pending = false;
      }
      if (pt == kRecStorer && !wait_flag_geq(flags + cur.u * 32 + 16, need, p.wait_ns)) timeout();
      if (role_any(NB, PIPE, failed)) break;
    }

    // ---- 2. elementwise: operand tiles; qd, kr^T and e^{g_last} straight into the record ----
    {
      if (PRE)
        prep::elementwise<true, true>(sm, gsum, gpre, dp, hq, rows, scale, gs + SR_QW, SR_KB, gs + SR_KRT,
                                      reinterpret_cast<float*>(gs + SR_GAM), rnorm, range_bad);
      else
        prep::elementwise<true, false>(sm, gsum, gpre, dp, hq, rows, scale, gs + SR_QW, SR_KB, gs + SR_KRT,
                                       reinterpret_cast<float*>(gs + SR_GAM), nullptr, range_bad);
    }
    fence_proxy_async_global();  // the record's plain stores, read by the chain's bulk copies
    if ((pt == 0 || pt == kRecStorer) && pub_pending) bulk_wait_group<0>();  // the previous record's stores have landed
    fence_proxy_async_smem();
    PSTAMP(3);
    role_sync(NB, PIPE);
    PSTAMP(4);
    if (pub_pending) {  // from warp 3 of the pipeline while warp 0 issues the MMAs
      if (pw == 3 && lane == 0) publish(pub_m, pub_u);
      pub_pending = false;
    }
    if (pt == kRecStorer) {  // qd to the record
      bulk_store(gs + SR_QW, sm + prep::QDS, 8192);
      bulk_store(gs + SR_QW + SR_KB, sm + prep::QDS + 8192, 8192);
      bulk_commit();
    }

    // ---- 3. the diagonal halves and the block below them of L and Aqk ----
    if (pw == 0) {
      tc_fence_after();
      prep::issue_lqk(tmem, D_PREP);
      umma_commit_warp(&bars[PB_PMMA]);
      ++pmma_issued;
    }
    if (next) prefetch_gb(nx, 0);
    __syncwarp();
    PSTAMP(5);
    if (mbar_wait(&bars[PB_PMMA], pmma_phase & 1, p.wait_ns)) ++pmma_phase;  // else still in flight: drained below
    else timeout();
    tc_fence_after();
    PSTAMP(6);

    // ---- 4. TMEM -> M (fp32), Aqk ----
    prep::readout_lqk(sm, tmem, beta_s, quad, cpart, lane);
    tc_fence_before();
    fence_proxy_async_smem();
    PSTAMP(7);
    if (role_any(NB, PIPE, failed)) break;
    PSTAMP(8);
    if (pt == 0) {
      bulk_store(gs + SR_AQK, sm + prep::AQK_STG, 8192);
      bulk_commit();
    }
    if (next) prefetch_gb(nx, 1);

    // ---- 5. inverse and A = T Diag(beta) ----
    prep::inverse_diag_blocks(sm, beta_s, pw, pt, lane);
    PSTAMP(9);
    role_sync(NB, PIPE);
    PSTAMP(10);
    if (next) prefetch_gb(nx, 2);
    if (pw < 3) inverse_block_columns(reinterpret_cast<float*>(sm + prep::MB), beta_s, sm + prep::AMAT, pw, lane);
    if (pt == 0) bulk_wait_read();  // the Aqk staging has been read: its buffer takes U^T next
    fence_proxy_async_smem();
    PSTAMP(11);
    role_sync(NB, PIPE);
    PSTAMP(12);

    // ---- 6. W = A kd (M = 64, kd as MN-major B) and U^T = v^T A^T (M = 128 value
    //         columns, v as MN-major A, A as K-major B) ----
    if (pw == 0) {
      if (!__any_sync(0xFFFFFFFFu, failed)) {
        tc_fence_after();
        constexpr uint32_t idesc_w = idesc_f16kind(64, 128) | IDESC_B_MN_MAJOR;
        constexpr uint32_t idesc_u = idesc_f16kind(128, 64) | IDESC_A_MN_MAJOR;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = D_PREP + ((prep::AMAT + ks * 32) >> 4);
          umma_f16_warp(tmem + TM_W, ad, D_KD_MN + ((ks * 2048) >> 4), idesc_w, ks != 0);
          umma_f16_warp(tmem + TM_U, D_V_MN + ((ks * 2048) >> 4), ad, idesc_u, ks != 0);
        }
        umma_commit_warp(&bars[PB_PMMA]);
        ++pmma_issued;
      }
    } else if (pt == kRecStorer && next && nx.m >= SRING) {
      // the next record's flow-control counter, read ahead while the products run (the
      // acquire load stalls this warp, which waits for the products anyway)
      flow_seen = ld_acquire_gpu(flags + nx.u * 32 + 16);
      flow_n = rn;
    }
    if (next) prefetch_gb(nx, 3);
    __syncwarp();
    PSTAMP(13);
    if (mbar_wait(&bars[PB_PMMA], pmma_phase & 1, p.wait_ns)) ++pmma_phase;  // else still in flight: drained below
    else timeout();
    tc_fence_after();
    PSTAMP(14);
    // the stacked tile (M and A by now) and v are free again: fetch the next record's tiles
    if (pt == 0 && next && !failed) issue_raw(nx, j + 1);

    // ---- 7. W -> staging over kd (bf16 SW128, warps 0-3), U^T -> staging over cA (warps
    //         4-7: row v of 64 tokens, 128-byte-swizzled) ----
    __syncwarp();
    if (cpart == 0) {
      const int i = 16 * quad + (lane & 15);
#pragma unroll
      for (int q2 = 0; q2 < 4; q2 += 2) {
        float r0[32], r1[32];
        tmem_ld32(tmem_addr(tmem, 32 * quad, TM_W + 32 * q2), r0);
        tmem_ld32(tmem_addr(tmem, 32 * quad, TM_W + 32 * (q2 + 1)), r1);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float* rr = h ? r1 : r0;
            const int q4 = q2 + h;
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8)
              st_v4(sm + prep::KDT + sw128_offset(i, 32 * q4 + 8 * j8, 64), pack2(rr[8 * j8], rr[8 * j8 + 1]),
                    pack2(rr[8 * j8 + 2], rr[8 * j8 + 3]), pack2(rr[8 * j8 + 4], rr[8 * j8 + 5]),
                    pack2(rr[8 * j8 + 6], rr[8 * j8 + 7]));
          }
        }
      }
    } else {
      const int v = 32 * quad + lane;
      uint8_t* row = sm + prep::USTG + v * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float rr[32];
        tmem_ld32(tmem_addr(tmem, 32 * quad, TM_U + 32 * h), rr);
        tmem_ld_wait();
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8)
          st_v4(row + (((4 * h + j8) ^ (v & 7)) << 4), pack2(rr[8 * j8], rr[8 * j8 + 1]),
                pack2(rr[8 * j8 + 2], rr[8 * j8 + 3]), pack2(rr[8 * j8 + 4], rr[8 * j8 + 5]),
                pack2(rr[8 * j8 + 6], rr[8 * j8 + 7]));
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    PSTAMP(15);
    if (role_any(NB, PIPE, failed)) break;
    PSTAMP(16);

    // ---- 8. W/U to the ring; published early in the next record (or at the end);
    //         a pipeline's first record goes out at once ----
    if (pt == 0) {
      bulk_store(gs + SR_QW + SR_W_IN_KB, sm + prep::KDT, 8192);
      bulk_store(gs + SR_QW + SR_KB + SR_W_IN_KB, sm + prep::KDT + 8192, 8192);
      bulk_store(gs + SR_U, sm + prep::USTG, 16384);
      bulk_commit();
      if (j == 0) bulk_wait_group<0>();
    }
    if (pt == kRecStorer && j == 0) bulk_wait_group<0>();  // (the first record is published below)
    pub_pending = true;
    pub_m = cur.m;
    pub_u = cur.u;
    if (j == 0) {
      role_sync(NB, PIPE);
      if (pw == 3 && lane == 0) publish(pub_m, pub_u);
      pub_pending = false;
    }
    PSTAMP(17);
    r = rn;
    cur = nx;
  }
  if (range_bad) atomicOr(p.status, kStatusRange);
  if (pt == 0 || pt == kRecStorer) bulk_wait_all();
  role_sync(NB, PIPE);
  if (pub_pending && pw == 3 && lane == 0 && !failed) publish(pub_m, pub_u);
  if (pt == 0) {  // drain what this pipeline issued
    if (raw_pending && !mbar_wait(&bars[PB_RAW], raw_pending_j & 1, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
    if (pmma_issued > pmma_phase && !mbar_wait(&bars[PB_PMMA], (pmma_issued - 1) & 1, DRAIN_LIMIT_NS))
      atomicOr(p.status, kStatusTimeout);
  }
  __syncwarp();
}

// --------------------------------------------------------------- chain ----
// The recurrence is carried transposed in TMEM (lanes = value columns v): S^T in fp32
// and as a bf16 copy, v_new^T in bf16, and the products [O^T | X^T] (two buffers, one
// per chunk parity).  The bf16 matrices are the A operands of the chain's MMAs; their B
// operands are the record's tiles in shared memory as the producer wrote them:
//   [O^T | X^T] = S^T [qd; W]^T      (N = 128, K = 128)
//   S^T += v_new^T kr                 (N = 128, K = 64)
//   O^T += v_new^T Aqk^T              (N = 64,  K = 64)
// with S^T scaled by e^{g_last} between chunks.  Warps 0-7 carry the recurrence: warp w
// reads TMEM lane quadrant w % 4 (v = 32 (w % 4) + lane) and takes half h = w / 4 of
// the other dimension (tokens 32 h + [0, 32) of v_new, key dims 64 h + [0, 64) of the
// state).  The next chunk's first product is issued as soon as these 8 warps have
// copied the state, into the other [O^T | X^T] buffer.  Warps 8-15 (same quadrants and
// halves) scale S^T for each chunk while its first product runs, emit the o rows one
// chunk behind, and (one lane) copy the records ahead.  The two groups meet only on named
// barriers that one side waits on and the other arrives at; each arrival of one group
// follows the other group's passage of that barrier's previous phase.
constexpr int kIssuerWarp = 0;     // issues every chain MMA (a recurrence warp)
constexpr int kLoader = 8 * 32;    // helper lane copying the records
constexpr int kStorer = 13 * 32;   // helper lane issuing the o tile stores
constexpr int CB_C = 4;            // [2] o product of a chunk (one barrier per [O^T | X^T] buffer)
// [2] per chunk parity: part B of the chunk's record has landed and its first product has
// completed (two arrivals: the copying lane's, with the bytes, and the product's commit)
constexpr int CB_AB = 6;
constexpr int CB_DRAIN = 8;        // every chain MMA issued has completed (end of the chain)
constexpr int kChainBars = 9;
static_assert(C_BAR + 8 * kChainBars <= C_MISC, "chain barriers stay below the tmem slot");
constexpr uint32_t NB_HELP = 5;    // named barrier of the 8 helper warps
constexpr uint32_t NB_SCALED = 6;  // recurrence warps wait (v_new stored), helper warps arrive (S^T scaled)
constexpr uint32_t NB_COPIED = 7;  // helper warps wait, recurrence warps arrive (bf16 copy of S^T taken)
constexpr uint32_t NB_OREAD = 8;   // recurrence warps wait, helper warps arrive (O^T of the chunk before read)
constexpr uint32_t TS = 0, TSB = 128, TVN = 192, TXO = 256;  // TMEM columns (TXO: two 128-column buffers)
// -DKDA_PROFILE: clock64 stamps of threads 0 and 256 of chain 0 at numbered points of
// one chunk, kept in shared memory (cheap enough not to disturb the timing)
#ifndef KDA_STAMP_CHUNK
#define KDA_STAMP_CHUNK 32
#endif
#ifdef KDA_PROFILE
#define STAMP(i)                                                                                 \
  do {                                                                                           \
    if (m == KDA_STAMP_CHUNK && u == 0 && (tid == 0 || tid == 256)) {                            \
      long long t_;                                                                              \
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(t_)::"memory");                               \
      *reinterpret_cast<volatile long long*>(sm + C_MISC + 64 + (tid ? 192 : 0) + 8 * (i)) = t_;  \
    }                                                                                            \
  } while (0)
#else
#define STAMP(i) \
  do {           \
  } while (0)
#endif

__device__ __forceinline__ void chain(const Maps& maps, const FwdParams& p, uint8_t* sm, uint32_t tmem, int u,
                                      uint32_t* flags) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;
  const bool rec = warp < 8;           // recurrence warp (else helper)
  const int h = (warp >> 2) & 1;       // half of the non-lane dimension
  const int vcol = 32 * quad + lane;   // this thread's value column
  const int HV = p.HV;
  const int ug = p.unit0 + u;          // the unit of the problem (u: of this launch)
  const int seq = ug / HV, hv = ug - seq * HV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C_BAR);
  long tok0;
  int len;
  seq_range(p, seq, tok0, len);
  const int NT = (len + C - 1) / C;
  uint8_t* ring = p.ring + static_cast<size_t>(u) * RING * GSLOT;
  uint32_t* ready = flags + u * 32;
  uint32_t* consumed = ready + 16;
  const uint32_t sb = smem_u32(sm);
  const uint64_t D_SW128 = sdesc_sw128(sb);
  auto d128 = [&](uint32_t off) { return D_SW128 + (off >> 4); };
  const uint32_t tl = tmem_addr(tmem, 32 * quad, 0);  // this warp's lane quadrant
  const size_t state_off = static_cast<size_t>(ug) * KD * VD;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  bool failed = false;
  int a_issued = 0, b_issued = 0, c_issued = 0;
  auto timeout = [&](int id, int at) {
    failed = true;
    atomicOr(p.status, kStatusTimeout);
#ifdef KDA_PROFILE
    atomicCAS(reinterpret_cast<unsigned long long*>(p.status) + 400, 0ull,
              (static_cast<unsigned long long>(blockIdx.x) << 40) | (static_cast<unsigned long long>(tid) << 24) |
                  (static_cast<unsigned long long>(at) << 8) | static_cast<unsigned long long>(id));
#endif
  };
  // a bounded wait, skipped once this thread has given up (the loop then runs to its end
  // without work, passing every named barrier the same number of times as the others)
  auto wait = [&](uint64_t* bar, uint32_t parity, int id, int at) {
    if (!failed && !mbar_wait(bar, parity, p.wait_ns)) timeout(id, at);
  };
  // Record copies by one helper lane into the buffers of the chunk finished last: part A
  // (three buffers) up to two chunks ahead, part B (two buffers) one chunk ahead.  The
  // lane learns that records are ready from acquire loads of the flags, eight ring slots
  // (one aligned 32-byte group) per load, so that the load's round trip to L2, which
  // stalls the warp, comes about once every eight chunks; part B of a record follows its
  // part A and needs no read of its own.  The producer fenced its stores to the async
  // proxy before publishing, so the copies need no fence.
  const bool is_loader = tid == kLoader;
  int next_a = 0, next_b = 0;  // first chunk whose part A / part B is not issued yet
  int known = 0;               // records [0, known) are known to be ready
  auto read_flags = [&]() {    // the group of ring slots holding record `known`, from it on
    const int s0 = known % SRING;
    uint32_t fv[8];
    ld_acquire_gpu_v8(ready + (s0 & ~7), fv);
    bool run = true;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j >= (s0 & 7) && run) {
        run = fv[j] >= static_cast<uint32_t>(known + 1);
        if (run) ++known;
      }
  };
  auto issue_a = [&](int n) {
    const int b = n % 3;
    mbar_arrive_expect_tx_relaxed(&bars[CB_FULL + b], REC_A_BYTES);
    bulk_load(sm + C_PA + b * PA_STRIDE, ring + static_cast<size_t>(n % SRING) * GSLOT, REC_A_BYTES, &bars[CB_FULL + b]);
#ifdef KDA_PROFILE
    if (u == 0 && n >= KDA_STAMP_M0 && n < KDA_STAMP_M0 + 64)
      reinterpret_cast<uint64_t*>(p.status)[264 + n - KDA_STAMP_M0] = globaltimer_ns();
#endif
  };
  auto issue_b = [&](int n) {
    const int b = n & 1;
    mbar_arrive_expect_tx_relaxed(&bars[CB_AB + b], PB_STRIDE);
    bulk_load(sm + C_PB + b * PB_STRIDE, ring + static_cast<size_t>(n % SRING) * GSLOT + SR_KRT, PB_STRIDE,
              &bars[CB_AB + b]);
#ifdef KDA_PROFILE
    if (u == 0 && n >= KDA_STAMP_M0 && n < KDA_STAMP_M0 + 64)
      reinterpret_cast<uint64_t*>(p.status)[330 + n - KDA_STAMP_M0] = globaltimer_ns();
#endif
  };
  auto pump_b = [&](int up_b) {
    while (next_b <= up_b && next_b < next_a) issue_b(next_b++);
  };
  // part A up to chunk up_a (waiting for the records up to must_a), then part B up to up_b
  auto pump = [&](int up_a, int must_a, int up_b) {
    while (!failed && next_a <= up_a && next_a < NT) {
      if (next_a >= known) read_flags();
      if (next_a >= known) {
        if (next_a > must_a) break;
        const uint64_t t0 = globaltimer_ns();
        while (next_a >= known && globaltimer_ns() - t0 <= p.wait_ns) read_flags();
        if (next_a >= known) {
          timeout(1, next_a);
          break;
        }
      }
      issue_a(next_a++);
    }
    if (!failed) pump_b(up_b);
  };
  // o rows of chunk mc from `ob` (bf16 pairs of tokens 2 t, 2 t + 1 of this thread's value
  // column): lane pairs (v, v + 1) swap halves, then the even lane stores the pair of value
  // columns for tokens 2 t and the odd lane for tokens 2 t + 1 (64 contiguous bytes per half-warp)
  auto store_o = [&](int mc, const uint32_t (&ob)[16]) {
    const int rows = min(C, len - mc * C);
    const bool odd = lane & 1;
    const int t0 = 32 * h + (odd ? 1 : 0);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + (static_cast<size_t>(tok0 + mc * C + t0) * HV + hv) * VD +
                                                (vcol & ~1));
    const size_t row2 = static_cast<size_t>(HV) * VD;  // two tokens, in 32-bit words
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, ob[t], 1);
      const uint32_t pairv = odd ? __byte_perm(got, ob[t], 0x7632) : __byte_perm(ob[t], got, 0x5410);
      if (t0 + 2 * t < rows) dst[t * row2] = pairv;
    }
  };
  // K-step ks (key dims 16 ks + [0, 16)) of [O^T | X^T] (buffer of chunk mc) = S^T [qd; W]^T
  auto issue_first_product_step = [&](int mc, int ks, bool first) {
    const uint32_t so = C_PA + (mc % 3) * PA_STRIDE;
    umma_f16_ts_warp(tmem + TXO + 128 * (mc & 1), tmem + TSB + 8 * ks, d128(so + SR_QW + (ks >> 2) * SR_KB + (ks & 3) * 32),
                     idesc_f16kind(128, 128), first ? 0u : 1u);
  };

  // Part A of chunk m + 1 is read at the end of chunk m (the next first product), part B
  // of chunk m from its start: during chunk m the lane must have issued part A of m + 1
  // and part B of m, and may issue part A of m + 2 and part B of m + 1.
  if (is_loader) pump(2, 0, 1);
  if (rec) {  // S^T and its bf16 copy from the initial state (key dims 64 h + [0, 64))
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float st[16];
      if (p.s0) {
        const float* src = p.s0 + state_off + vcol;
#pragma unroll
        for (int i = 0; i < 16; ++i) st[i] = src[static_cast<size_t>(64 * h + 16 * j + i) * VD];
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) st[i] = 0.f;
      }
      uint32_t hb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) hb[i] = pack2(st[2 * i], st[2 * i + 1]);
      tmem_st8u(tl + TSB + 32 * h + 8 * j, hb);
      tmem_st16(tl + TS + 64 * h + 16 * j, st);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  role_sync(NB_CHAIN_ALL, NTHREADS);
  tc_fence_after();
  if (warp == kIssuerWarp && NT > 0) {  // the first chunk's first product
    if (!mbar_wait(&bars[CB_FULL], 0, p.wait_ns)) timeout(4, 0);  // part A of chunk 0
    __syncwarp();
    if (!__any_sync(0xFFFFFFFFu, failed)) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) issue_first_product_step(0, ks, ks == 0);
      umma_commit_warp(&bars[CB_AB]);
      ++a_issued;
    }
  }

#ifdef KDA_PROFILE
  if (tid == 0 && u == 0) reinterpret_cast<uint64_t*>(p.status)[127] = globaltimer_ns();
#endif
  if (rec) {
    for (int m = 0; m < NT; ++m) {
      const int s = m & 1;
      const uint32_t sbb = C_PB + s * PB_STRIDE - SR_KRT;  // part B of this chunk (record offsets)
      const bool more = m + 1 < NT;
      STAMP(0);
      // ---- v_new^T = U^T - X^T: tokens 32 h + [0, 32) of this thread's value column ----
      wait(&bars[CB_AB + s], (m >> 1) & 1, 6, m);  // part B landed, X^T computed
      const uint8_t* urow = sm + sbb + SR_U + vcol * 128;  // U^T row v (64 tokens, 128-byte-swizzled)
      __syncwarp();
      tc_fence_after();
      STAMP(2);
      {
        const uint32_t txt = TXO + 128 * s + 64;  // X^T of this chunk
        float xv[32];
        tmem_ld16(tl + txt + 32 * h, reinterpret_cast<float(&)[16]>(xv[0]));
        tmem_ld16(tl + txt + 32 * h + 16, reinterpret_cast<float(&)[16]>(xv[16]));
        uint4 uu[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) uu[i] = *reinterpret_cast<const uint4*>(urow + (((4 * h + i) ^ (vcol & 7)) << 4));
        tmem_ld_wait();
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {  // tokens 32 h + 16 q2 + [0, 16)
          const uint32_t uw[8] = {uu[2 * q2].x, uu[2 * q2].y, uu[2 * q2].z, uu[2 * q2].w,
                                  uu[2 * q2 + 1].x, uu[2 * q2 + 1].y, uu[2 * q2 + 1].z, uu[2 * q2 + 1].w};
          uint32_t vn[8];
#pragma unroll
          for (int t = 0; t < 8; ++t)
            vn[t] = pack2(__uint_as_float(uw[t] << 16) - xv[16 * q2 + 2 * t],
                          __uint_as_float(uw[t] & 0xFFFF0000u) - xv[16 * q2 + 2 * t + 1]);
          tmem_st8u(tl + TVN + 16 * h + 8 * q2, vn);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      STAMP(3);
      named_bar_sync(NB_SCALED, NTHREADS);  // v_new^T stored; the helpers have scaled S^T
      STAMP(4);
      if (warp == kIssuerWarp && !__any_sync(0xFFFFFFFFu, failed)) {  // S^T += v_new^T kr, O^T += v_new^T Aqk^T
        tc_fence_after();
        constexpr uint32_t kstep[4] = {0, 2, 4, 6};  // 32-byte K steps inside a 128-byte swizzled row
        umma_ts_chain<4>(tmem + TS, tmem + TVN, d128(sbb + SR_KRT), kstep, idesc_f16kind(128, 128), 1u);
        umma_commit_warp(&bars[CB_B]);
        ++b_issued;
        if (!p.h)  // (the state pass keeps the commit, so the barrier's phases stay in step)
          umma_ts_chain<4>(tmem + TXO + 128 * s, tmem + TVN, d128(sbb + SR_AQK), kstep, idesc_f16kind(128, 64), 1u);
        umma_commit_warp(&bars[CB_C + s]);
        ++c_issued;
        if (lane == 0) st_relaxed_gpu(consumed, static_cast<uint32_t>(m + 1));  // record m is in shared memory
      }
      if (warp == kIssuerWarp && more)  // part A of the next chunk (copied a chunk ago), while MMA_b runs
        wait(&bars[CB_FULL + (m + 1) % 3], ((m + 1) / 3) & 1, 4, m + 1);
      STAMP(5);
      // ---- bf16 copy of S^T, then the next chunk's first product into the other buffer ----
      wait(&bars[CB_B], m & 1, 9, m);
      __syncwarp();
      tc_fence_after();
      STAMP(6);
      if (more) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float sv[32];
          tmem_ld32(tl + TS + 64 * h + 32 * j, sv);
          tmem_ld_wait();
          uint32_t hb[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) hb[i] = pack2(sv[2 * i], sv[2 * i + 1]);
          tmem_st16u(tl + TSB + 32 * h + 16 * j, hb);
        }
        tmem_st_wait();
        tc_fence_before();
        // the copy is complete, and the helpers have read O^T of chunk m - 1 from the buffer
        // the next first product overwrites; only then may the helpers go on to the next
        // chunk (scaling S^T for it), so that they never arrive at a named barrier before
        // the recurrence warps have left its previous phase
        named_bar_sync(NB_OREAD, NTHREADS);
        named_bar_arrive(NB_COPIED, NTHREADS);
        if (warp == kIssuerWarp) {
          __syncwarp();
          if (!__any_sync(0xFFFFFFFFu, failed)) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) issue_first_product_step(m + 1, ks, ks == 0);
            umma_commit_warp(&bars[CB_AB + (s ^ 1)]);
            ++a_issued;
          }
        }
      }
      STAMP(7);
    }
  } else {
    // ---- helpers, one step behind on the o rows: in step m the state scale of chunk m,
    //      then the o rows of chunk m - 1 (its o product has completed; the buffer is
    //      rewritten by the first product of chunk m + 1, issued after the arrival below),
    //      then the record copies ----
    auto emit_o = [&](int mc) {
      wait(&bars[CB_C + (mc & 1)], (mc >> 1) & 1, 11, mc);
      if (p.h) return;  // state pass: no output (every helper returns here alike)
      __syncwarp();
      tc_fence_after();
      const uint32_t tot = TXO + 128 * (mc & 1);  // O^T of this chunk
      const int rows = min(C, len - mc * C);
      if (rows == C) {
        // o^T tiles to the staging buffer as [token][v] rows (8x8 blocks transposed by
        // stmatrix; 128-byte swizzle, two 64-column halves), then two TMA tile stores
        uint8_t* stage = sm + C_STG + (mc & 1) * 16384;
        const int mi = lane >> 3, mr = lane & 7;  // the matrix and row this lane addresses
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // tokens 32 h + 8 j + [0, 8)
          uint32_t a[4], b[4];
          tmem_ld_16x256b(tmem_addr(tmem, 32 * quad, tot + 32 * h + 8 * j), a);
          tmem_ld_16x256b(tmem_addr(tmem, 32 * quad + 16, tot + 32 * h + 8 * j), b);
          tmem_ld_wait();
          const int c = 32 * h + 8 * j + mr, v = 32 * quad + 8 * mi;
          stmatrix_x4_trans(smem_u32(stage + (v >> 6) * 8192 + c * 128 + ((((v & 63) >> 3) ^ (c & 7)) << 4)),
                            pack2(__uint_as_float(a[0]), __uint_as_float(a[1])),
                            pack2(__uint_as_float(a[2]), __uint_as_float(a[3])),
                            pack2(__uint_as_float(b[0]), __uint_as_float(b[1])),
                            pack2(__uint_as_float(b[2]), __uint_as_float(b[3])));
        }
        fence_proxy_async_smem();
        role_sync(NB_HELP, 256);
        if (tid == kStorer && !failed) {
          const int row0 = static_cast<int>(tok0) + mc * C;
          tma_store_3d(&maps.o, stage, 0, hv, row0);
          tma_store_3d(&maps.o, stage + 8192, 64, hv, row0);
          bulk_commit();
          bulk_wait_group_read<1>();  // the previous chunk's tiles have been read: its buffer is free
        }
      } else {  // a sequence's partial last chunk: plain stores of its rows
        uint32_t ob[16];  // bf16 pairs (tokens 2 t, 2 t + 1) of this thread's value column
        float ov[32];
        tmem_ld32(tl + tot + 32 * h, ov);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 16; ++t) ob[t] = pack2(ov[2 * t], ov[2 * t + 1]);
        if (!failed) store_o(mc, ob);
      }
    };
    for (int m = 0; m <= NT; ++m) {
      const uint32_t sa = C_PA + (m % 3) * PA_STRIDE;  // part A of this chunk
      STAMP(0);
      if (m < NT) {
        // ---- helpers: S^T <- S^T Diag(e^{g_last}) (key dims 64 h + [0, 64)) while the first
        //      product runs (it reads the bf16 copy), once the previous chunk's state copy is
        //      done (its state product completed before) ----
        if (m > 0) named_bar_sync(NB_COPIED, NTHREADS);
        tc_fence_after();
        // part B of the next chunk (its record is known ready) into the buffer of chunk m - 1:
        // that chunk's v_new preceded its state copy and its state product completed before
        // it; its o product, which reads Aqk there, is waited for here
        if (is_loader) {
          if (m > 0) wait(&bars[CB_C + ((m - 1) & 1)], ((m - 1) >> 1) & 1, 11, m - 1);
          pump_b(m + 1);
        }
        wait(&bars[CB_FULL + m % 3], (m / 3) & 1, 4, m);
        // state pass: the bf16 copy of S^T (the state entering chunk m, as the chain's MMAs
        // read it; rewritten only by this chunk's state copy, after the arrival below),
        // key dims 64 h + [0, 64) of value column vcol as 32 bf16 pairs along k
        uint32_t hs[32];
        if (p.h) {
          tmem_ld32(tl + TSB + 32 * h, reinterpret_cast<float(&)[32]>(hs));
          tmem_ld_wait();
        }
        {
          const float* gam = reinterpret_cast<const float*>(sm + sa + SR_GAM) + 64 * h;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float sv[16];
            tmem_ld16(tl + TS + 64 * h + 16 * j, sv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 g = reinterpret_cast<const float4*>(gam + 16 * j)[i];
              sv[4 * i] *= g.x;
              sv[4 * i + 1] *= g.y;
              sv[4 * i + 2] *= g.z;
              sv[4 * i + 3] *= g.w;
            }
            tmem_st16(tl + TS + 64 * h + 16 * j, sv);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        named_bar_arrive(NB_SCALED, NTHREADS);
        STAMP(1);
        if (p.h) {
          // h[m] rows k = 64 h + 2c, 2c + 1: lane pairs (v, v + 1) swap their words, then the
          // even lane stores (S[2c][v], S[2c][v + 1]) and the odd lane (S[2c+1][v - 1], S[2c+1][v])
          // (64 contiguous bytes per half-warp and store)
          const bool odd = lane & 1;
          uint16_t* hb = p.h + ((static_cast<size_t>(seq) * HV + hv) * p.h_chunks + m) * KD * VD + (vcol & ~1);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint32_t t = __shfl_xor_sync(0xFFFFFFFFu, hs[c], 1);
            const int kk = 64 * h + 2 * c + (odd ? 1 : 0);
            *reinterpret_cast<uint32_t*>(hb + static_cast<size_t>(kk) * VD) =
                odd ? __byte_perm(t, hs[c], 0x7632) : __byte_perm(hs[c], t, 0x5410);
          }
        }
      }
      if (m > 0) {
        if (m == NT) role_sync(NB_HELP, 256);  // the storer's last wait precedes the staging writes
        emit_o(m - 1);
      }
      if (m + 1 < NT) {
        tc_fence_before();
        named_bar_arrive(NB_OREAD, NTHREADS);
      }
      // part A of chunk m + 2 into the buffer of chunk m - 1 (free, as above)
      if (is_loader && m < NT) pump(m + 2, m + 1, m + 1);
      STAMP(8);
    }
  }
  if (warp == kIssuerWarp && a_issued + b_issued + c_issued > 0) {  // MMAs still in flight after a failure
    umma_commit_warp(&bars[CB_DRAIN]);
    if (lane == 0 && !mbar_wait(&bars[CB_DRAIN], 0, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
  }
#ifdef KDA_PROFILE
  __syncwarp();
  if (u == 0 && (tid == 0 || tid == 256)) {  // the stamps of chunk KDA_STAMP_CHUNK
    const long long* st = reinterpret_cast<const long long*>(sm + C_MISC + 64 + (tid ? 192 : 0));
    for (int i = 0; i < 24; ++i) reinterpret_cast<long long*>(p.status)[432 + (tid ? 24 : 0) + i] = st[i];
  }
#endif
  if (is_loader) {  // copies still in flight after an abort (a consumed phase returns at once)
    for (int n = max(0, next_a - 3); n < next_a; ++n)
      if (!mbar_wait(&bars[CB_FULL + n % 3], (n / 3) & 1, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
    for (int n = max(0, next_b - 2); n < next_b; ++n)  // (after a failure the phase may lack its commit)
      if (!mbar_wait(&bars[CB_AB + (n & 1)], (n >> 1) & 1, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
  }
  if (tid == kStorer) bulk_wait_all();
  __syncwarp();
  if (rec && p.sfin && !failed) {  // S^T -> final state (for each k a warp writes 128 contiguous bytes)
    tc_fence_after();
    float* dst = p.sfin + state_off + vcol;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float sv[32];
      tmem_ld32(tl + TS + 64 * h + 32 * j, sv);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[static_cast<size_t>(64 * h + 32 * j + i) * VD] = sv[i];
    }
  }
}
}  // namespace split

template <bool PRE>
__global__ void __launch_bounds__(split::NTHREADS, 1)
kda_chunk_split_kernel(const __grid_constant__ Maps maps, const FwdParams p, int NU, int NREC) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool is_chain = static_cast<int>(blockIdx.x) < NU;
  uint32_t* flags = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.status) + kFlagOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + split::TMEM_SLOT);
#ifdef KDA_PROFILE
  // [120] entry of CTA 0, [121] entry of the first producer CTA, [122] the last CTA's exit,
  // [123] chain 0's exit, [124] the last producer's exit
  if (tid == 0 && (blockIdx.x == 0 || static_cast<int>(blockIdx.x) == NU))
    reinterpret_cast<uint64_t*>(p.status)[blockIdx.x == 0 ? 120 : 121] = globaltimer_ns();
#endif
  if (tid == 0) {
    if (is_chain) {
      uint64_t* cb = reinterpret_cast<uint64_t*>(sm + split::C_BAR);
      for (int i = 0; i < split::kChainBars; ++i)  // CB_FULL[3], CB_B, CB_C[2], CB_AB[2], CB_DRAIN
        mbar_init(&cb[i], i == split::CB_AB || i == split::CB_AB + 1 ? 2 : 1);
      if (!p.h) tma_prefetch_desc(&maps.o);
    } else {
      for (int pp = 0; pp < 2; ++pp) {
        uint64_t* pb = reinterpret_cast<uint64_t*>(sm + pp * split::P_STRIDE + split::P_BAR);
        mbar_init(&pb[split::PB_RAW], 1);
        mbar_init(&pb[split::PB_PMMA], 1);
      }
      tma_prefetch_desc(&maps.q32);
      tma_prefetch_desc(&maps.k32);
      tma_prefetch_desc(&maps.v);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
#ifdef KDA_PROFILE
  // [119] the first producer CTA past its TMEM allocation and the block barrier
  if (tid == 0 && static_cast<int>(blockIdx.x) == NU) reinterpret_cast<uint64_t*>(p.status)[119] = globaltimer_ns();
#endif
  if (is_chain) {
    split::chain(maps, p, sm, tmem, static_cast<int>(blockIdx.x), flags);
  } else {  // records r = m NU + u, strided over the producer pipelines
    const int pipe = tid >> 8;
    const int pb = static_cast<int>(blockIdx.x) - NU;
    const int NQ = 2 * (static_cast<int>(gridDim.x) - NU);
    split::producer<PRE>(maps, p, sm + pipe * split::P_STRIDE, tmem + 256u * static_cast<uint32_t>(pipe), pipe,
                    2 * pb + pipe, NQ, NU, NREC, flags);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
#ifdef KDA_PROFILE
  if (tid == 0) {
    const unsigned long long t = globaltimer_ns();
    unsigned long long* w = reinterpret_cast<unsigned long long*>(p.status);
    atomicMax(w + 122, t);
    if (blockIdx.x == 0) w[123] = t;
    if (!is_chain) atomicMax(w + 124, t);
  }
#endif
}

// ======================================================================
// Parallel output kernel: o of every chunk from the state entering it.
//
// With h[n] (the state entering chunk n, from the state pass) the chunks no longer
// depend on each other:  o_n = qd_n h[n] + Aqk_n (U_n - W_n h[n])  (the a8 output of the
// chunked form with its a7 v_new, page "手撕KDA", section "1 Naive"; the per-chunk
// states of the C++ port in section 1.1).  One CTA of 8 warps per (chunk, value head,
// sequence), two per SM: it prepares the chunk as a producer pipeline does (the prep::
// steps: elementwise pass, the L/Aqk product, the inverse, W = A kd and U = A v), loads
// h[n] (bf16, MN-major) over the stacked tile those steps no longer need, and runs
//   X = W h[n] (M = 64, N = 128, K = 128),  v_new = U - X (bf16, over the raw v tile),
//   O = qd h[n] + Aqk v_new (M = 64, N = 128, K = 128 then 64)
// with fp32 accumulators in TMEM.  Waits are bounded (p.wait_ns); a timed-out wait
// sets kStatusTimeout, later products are not issued, and what was issued is drained.
// ======================================================================
namespace outk {
constexpr int NTHREADS = 256;
constexpr uint32_t O_BETA = prep::QDS + 16384, O_GSUM = O_BETA + 256, O_BAR = O_GSUM + 2048;
constexpr uint32_t O_MISC = O_BAR + 64, SMEM_BYTES = O_MISC + 64, SMEM_ALLOC = SMEM_BYTES + 1024;
static_assert(2 * SMEM_ALLOC <= 232448, "two output CTAs per SM");
constexpr int OB_RAW = 0, OB_MMA = 1, OB_H = 2;
constexpr uint32_t TM_W = 0, TM_U = 128, TM_X = 0, TM_O = 128, TMEM_COLS = 256;
constexpr uint32_t H_TX = 32768;

struct Maps {
  CUtensorMap q32, k32, v;  // as the chunk kernels'
  CUtensorMap h;            // h as [rows of 128 value columns], (64, 128) boxes
};
}  // namespace outk

__global__ void __launch_bounds__(outk::NTHREADS, 2)
kda_chunk_output_kernel(const __grid_constant__ outk::Maps maps, const FwdParams p) {
  using namespace outk;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + O_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + O_MISC);
  float* beta_s = reinterpret_cast<float*>(sm + O_BETA);
  float* gsum = reinterpret_cast<float*>(sm + O_GSUM);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pt = tid, dp = pt & 63, hq = pt >> 6, quad = warp & 3, cpart = warp >> 2;
  const int m = blockIdx.x, hv = blockIdx.y, seq = blockIdx.z;
  const int HV = p.HV, hk = hv / (HV / p.H);
  const long tok0 = static_cast<long>(seq) * p.T + static_cast<long>(m) * C;
  const int rows = min(C, p.T - m * C);

  if (tid == 0) {
    mbar_init(&bars[OB_RAW], 1);
    mbar_init(&bars[OB_MMA], 1);
    mbar_init(&bars[OB_H], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, outk::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sb = smem_u32(sm);
  const uint64_t D_PREP = sdesc_sw128(sb);
  auto d128 = [&](uint32_t off) { return D_PREP + (off >> 4); };
  const uint64_t D_KD_MN = sdesc(sb + prep::KDT, 8192, 1024, 2);
  const uint64_t D_V_MN = sdesc(sb + prep::VRAW, 8192, 1024, 2);  // raw v, then v_new
  const uint64_t D_H_MN = sdesc(sb + prep::QK, 16384, 1024, 2);   // h[n]: key dims as K, value columns as N
  bool failed = false, raw_issued = false, h_issued = false;
  uint32_t mma_issued = 0, mma_done = 0;
  auto mma_wait = [&]() {  // all threads: the products issued so far have completed
    if (!failed) {
      if (mbar_wait(&bars[OB_MMA], mma_done & 1, p.wait_ns)) ++mma_done;
      else { failed = true; atomicOr(p.status, kStatusTimeout); }
    }
    tc_fence_after();
  };

  // ---- 1. raw tiles (TMA), g and beta (registers) ----
  if (tid == 0) {
    prep::issue_raw(sm, &maps.q32, &maps.k32, &maps.v, &bars[OB_RAW], hk, hv, static_cast<int>(tok0));
    raw_issued = true;
  }
  float2 g[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int c = 16 * hq + i;
    g[i] = (c < rows) ? __ldg(reinterpret_cast<const float2*>(p.g + (static_cast<size_t>(tok0 + c) * HV + hv) * KD) + dp)
                      : make_float2(0.f, 0.f);
  }
  if (pt < C) beta_s[pt] = (pt < rows) ? __ldg(p.beta + static_cast<size_t>(tok0 + pt) * HV + hv) : 0.f;
  {
    float2 qsum = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      qsum.x += g[i].x;
      qsum.y += g[i].y;
    }
    reinterpret_cast<float2*>(gsum + hq * KD)[dp] = qsum;
  }
  if (!mbar_wait(&bars[OB_RAW], 0, p.wait_ns)) {
    failed = true;
    atomicOr(p.status, kStatusTimeout);
  }
  failed = __syncthreads_or(failed);

  // ---- 2. elementwise pass (qd to its tile; no record) ----
  bool range_bad = false;
  if (!failed)
    prep::elementwise<true, false, false>(sm, gsum, g, dp, hq, rows, p.scale, sm, 0, sm, reinterpret_cast<float*>(sm), nullptr,
                                          range_bad);
  if (range_bad) atomicOr(p.status, kStatusRange);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- 3. L and Aqk; readout ----
  if (warp == 0 && !failed) {
    prep::issue_lqk(tmem, D_PREP);
    umma_commit_warp(&bars[OB_MMA]);
    ++mma_issued;
  }
  mma_wait();
  if (!failed) prep::readout_lqk(sm, tmem, beta_s, quad, cpart, lane);
  tc_fence_before();
  fence_proxy_async_smem();
  failed = __syncthreads_or(failed);

  // ---- 4. T = (I + M)^{-1}, A = T Diag(beta) ----
  if (!failed) prep::inverse_diag_blocks(sm, beta_s, warp, pt, lane);
  __syncthreads();
  if (!failed && warp < 3) inverse_block_columns(reinterpret_cast<float*>(sm + prep::MB), beta_s, sm + prep::AMAT, warp, lane);
  fence_proxy_async_smem();
  __syncthreads();

  // ---- 5. W = A kd, U = A v ----
  if (tid == 0 && !failed) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_f16kind(64, 128) | IDESC_B_MN_MAJOR;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t ad = d128(prep::AMAT + ks * 32);
      umma_f16(tmem + outk::TM_W, ad, D_KD_MN + ((ks * 2048) >> 4), idesc, ks != 0);
      umma_f16(tmem + outk::TM_U, ad, D_V_MN + ((ks * 2048) >> 4), idesc, ks != 0);
    }
    umma_commit(&bars[OB_MMA]);
    ++mma_issued;
  }
  mma_wait();
  // h[n] over the stacked tile (M and A are no longer read)
  if (tid == 0 && !failed) {
    const int hrow = ((seq * HV + hv) * p.h_chunks + m) * KD;
    mbar_arrive_expect_tx(&bars[OB_H], H_TX);
    tma_load_2d(sm + prep::QK, &maps.h, &bars[OB_H], 0, hrow);
    tma_load_2d(sm + prep::QK + 16384, &maps.h, &bars[OB_H], 64, hrow);
    h_issued = true;
  }
  // W -> bf16 K-major tile over kd (the A operand of X = W h)
  if (!failed) {
    const int i = 16 * quad + (lane & 15);
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      float r[32];
      tmem_ld32(tmem_addr(tmem, 32 * quad, outk::TM_W + 64 * cpart + 32 * q2), r);
      tmem_ld_wait();
      if (lane < 16) {
        const int c0 = 64 * cpart + 32 * q2;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8)
          st_v4(sm + prep::KDT + sw128_offset(i, c0 + 8 * j8, 64), pack2(r[8 * j8], r[8 * j8 + 1]),
                pack2(r[8 * j8 + 2], r[8 * j8 + 3]), pack2(r[8 * j8 + 4], r[8 * j8 + 5]),
                pack2(r[8 * j8 + 6], r[8 * j8 + 7]));
      }
    }
  }
  tc_fence_before();
  fence_proxy_async_smem();
  __syncthreads();

  // ---- 6. X = W h[n] ----
  if (!failed && h_issued && !mbar_wait(&bars[OB_H], 0, p.wait_ns)) {
    failed = true;
    atomicOr(p.status, kStatusTimeout);
  }
  if (tid == 0 && !failed) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_f16kind(64, 128) | IDESC_B_MN_MAJOR;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_f16(tmem + outk::TM_X, d128(prep::KDT + kb * 8192 + ks * 32), D_H_MN + (((kb * 4 + ks) * 2048) >> 4), idesc,
                 (kb | ks) != 0);
    umma_commit(&bars[OB_MMA]);
    ++mma_issued;
  }
  failed = __syncthreads_or(failed);
  mma_wait();

  // ---- 7. v_new = U - X as bf16 over the raw v tile (MN-major: rows = tokens) ----
  if (!failed) {
    const int i = 16 * quad + (lane & 15);
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      const int c0 = 64 * cpart + 32 * q2;
      float ur[32], xr[32];
      tmem_ld32(tmem_addr(tmem, 32 * quad, outk::TM_U + c0), ur);
      tmem_ld32(tmem_addr(tmem, 32 * quad, outk::TM_X + c0), xr);
      tmem_ld_wait();
      if (lane < 16) {
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          const int c = c0 + 8 * j8;
          st_v4(sm + prep::VRAW + (c >> 6) * 8192 + sw128_offset(i, c & 63, 64),
                pack2(ur[8 * j8] - xr[8 * j8], ur[8 * j8 + 1] - xr[8 * j8 + 1]),
                pack2(ur[8 * j8 + 2] - xr[8 * j8 + 2], ur[8 * j8 + 3] - xr[8 * j8 + 3]),
                pack2(ur[8 * j8 + 4] - xr[8 * j8 + 4], ur[8 * j8 + 5] - xr[8 * j8 + 5]),
                pack2(ur[8 * j8 + 6] - xr[8 * j8 + 6], ur[8 * j8 + 7] - xr[8 * j8 + 7]));
        }
      }
    }
  }
  tc_fence_before();
  fence_proxy_async_smem();
  __syncthreads();

  // ---- 8. O = qd h[n] + Aqk v_new (over U's columns, read by now) ----
  if (tid == 0 && !failed) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_f16kind(64, 128) | IDESC_B_MN_MAJOR;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_f16(tmem + outk::TM_O, d128(prep::QDS + kb * 8192 + ks * 32), D_H_MN + (((kb * 4 + ks) * 2048) >> 4), idesc,
                 (kb | ks) != 0);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_f16(tmem + outk::TM_O, d128(prep::AQK_STG + ks * 32), D_V_MN + ((ks * 2048) >> 4), idesc, 1u);
    umma_commit(&bars[OB_MMA]);
    ++mma_issued;
  }
  mma_wait();

  // ---- 9. o rows (bf16) ----
  if (!failed) {
    const int i = 16 * quad + (lane & 15);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      const int c0 = 64 * cpart + 32 * q2;
      float r[32];
      tmem_ld32(tmem_addr(tmem, 32 * quad, outk::TM_O + c0), r);
      tmem_ld_wait();
      if (lane < 16 && i < rows) {
        uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(tok0 + i) * HV + hv) * VD + c0);
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8)
          dst[j8] = make_uint4(pack2(r[8 * j8], r[8 * j8 + 1]), pack2(r[8 * j8 + 2], r[8 * j8 + 3]),
                               pack2(r[8 * j8 + 4], r[8 * j8 + 5]), pack2(r[8 * j8 + 6], r[8 * j8 + 7]));
      }
    }
  }

  // drain what was issued before releasing the memory it touches
  if (tid == 0) {
    if (raw_issued && !mbar_wait(&bars[OB_RAW], 0, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
    if (h_issued && !mbar_wait(&bars[OB_H], 0, DRAIN_LIMIT_NS)) atomicOr(p.status, kStatusTimeout);
    if (mma_issued > mma_done && !mbar_wait(&bars[OB_MMA], (mma_issued - 1) & 1, DRAIN_LIMIT_NS))
      atomicOr(p.status, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, outk::TMEM_COLS);
}

// ------------------------------------------------------------------ host ----
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D map over a [tokens, heads, dim] bf16 tensor with a (64, 1, box_tokens) box, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int dim, int heads, long tokens, int box_tokens = C) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dim) * 2, static_cast<cuuint64_t>(heads) * dim * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_tokens)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over h as rows of 128 bf16 value columns, (64, 128) boxes, 128-byte swizzle.
bool make_map_h(CUtensorMap* m, const void* base, long rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(VD), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(VD) * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

static_assert(static_cast<size_t>(tc::RING) * tc::GSLOT == kRingBytesPerUnit, "ring layout");

// The parallel output kernel: one CTA per (chunk, value head, sequence); fixed-length
// sequences (p.cu == nullptr), p.h holding p.h_chunks states per (sequence, value head).
cudaError_t launch_chunk_output(const FwdParams& p, cudaStream_t stream) {
  static std::mutex mu;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && !attr[dev]) {
      const cudaError_t e = cudaFuncSetAttribute(tc::kda_chunk_output_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, tc::outk::SMEM_ALLOC);
      if (e != cudaSuccess) return e;
      attr[dev] = true;
    }
  }
  const long tokens = static_cast<long>(p.num_seqs) * p.T;
  tc::outk::Maps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!tc::make_map(&maps.q32, p.q, tc::KD, p.H, tokens, 32) || !tc::make_map(&maps.k32, p.k, tc::KD, p.H, tokens, 32) ||
      !tc::make_map(&maps.v, p.v, tc::VD, p.HV, tokens) ||
      !tc::make_map_h(&maps.h, p.h, static_cast<long>(p.num_seqs) * p.HV * p.h_chunks * tc::KD))
    return cudaErrorInvalidValue;
  if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream) != cudaSuccess) return cudaGetLastError();
  const dim3 grid(p.h_chunks, p.HV, p.num_seqs);
  tc::kda_chunk_output_kernel<<<grid, tc::outk::NTHREADS, tc::outk::SMEM_ALLOC, stream>>>(maps, p);
  return cudaGetLastError();
}

size_t chunk_tc_ring_bytes(int num_seqs, int HV) {
  return static_cast<size_t>(num_seqs) * HV * tc::RING * tc::GSLOT;
}

bool chunk_tc_supported(const FwdParams& p, bool bf16) {
  const long tokens = p.cu ? static_cast<long>(p.T) : static_cast<long>(p.num_seqs) * p.T;
  return bf16 && p.K == tc::KD && p.V == tc::VD && tokens > 0 && tc::encoder() != nullptr;
}

namespace {
// Which chunk kernel runs: the split kernel (chain and producer roles on separate
// SMs) when the units are few enough to leave three quarters of the SMs to the
// producers, else the cluster kernel.  KDA_CHUNK_SPLIT=0 or 1 in the environment
// forces one of them (1 still needs a unit count the split kernel can hold).
int split_override() {
  const char* e = std::getenv("KDA_CHUNK_SPLIT");
  return e ? std::atoi(e) : -1;
}
struct DeviceInfo {
  int sms = 0;
  bool coop = false, split_fits = false;
  bool fused_attr = false;  // the cluster kernel's shared-memory attribute is set on this device
};
const DeviceInfo& device_info() {
  static std::mutex mu;
  static DeviceInfo info[64];
  static bool known[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!known[dev]) {
    DeviceInfo& d = info[dev];
    int coop = 0;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    d.coop = coop != 0;
    d.split_fits = true;
    for (auto kern : {tc::kda_chunk_split_kernel<false>, tc::kda_chunk_split_kernel<true>}) {
      int blocks = 0;
      d.split_fits = d.split_fits &&
                     cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::split::SMEM_ALLOC) ==
                         cudaSuccess &&
                     cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, tc::split::NTHREADS,
                                                                   tc::split::SMEM_ALLOC) == cudaSuccess &&
                     blocks >= 1;
    }
    d.fused_attr = true;
    for (auto kern : {tc::kda_chunk_fused_kernel<false>, tc::kda_chunk_fused_kernel<true>})
      d.fused_attr = d.fused_attr && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                          tc::SMEM_ALLOC) == cudaSuccess;
    cudaGetLastError();
    known[dev] = true;
  }
  return info[dev];
}
}  // namespace

// How the split kernel covers the NS x HV (sequence, value head) units, of about `chunks`
// chunks each, on the current device: `launches` stream-ordered launches of at most
// `per_launch` consecutive units (their chains take one SM each; automatic plans leave
// three quarters of the SMs to the producers), or launches == 0 when the cluster kernel
// runs instead.  A launch takes whole sequences where a sequence's heads fit one.  More
// units than one launch holds pay a launch's start (~20 us before its chains have
// records) per launch, which long sequences amortise: problems with at least
// kMinBatchedChunks chunks per sequence (on average) run as several launches.  With
// packed sequences a launch lasts as long as its longest one, so they take that path
// only when a launch holds one sequence (HV > cap / 2); other packed problems with more
// units, and shorter ones, run the cluster kernel.
constexpr long kMinBatchedChunks = 16;
struct SplitPlan {
  int launches = 0, per_launch = 0;
};
SplitPlan split_plan(int NS, int HV, long chunks, bool packed) {
  const DeviceInfo& dev = device_info();
  const int mode = split_override();
  const int NU = NS * HV;
  SplitPlan plan;
  if (!dev.coop || !dev.split_fits || mode == 0 || NU < 1) return plan;
  const int cap = std::min(kMaxSplitUnits, mode == 1 ? dev.sms - 2 : dev.sms / 4);
  if (cap < 1 || (NU > cap && mode != 1 && ((packed && 2 * HV <= cap) || chunks < kMinBatchedChunks))) return plan;
  if (HV <= cap) {  // whole sequences per launch, spread evenly
    const int seqs_cap = cap / HV;
    plan.launches = (NS + seqs_cap - 1) / seqs_cap;
    plan.per_launch = ((NS + plan.launches - 1) / plan.launches) * HV;
  } else {
    plan.launches = (NU + cap - 1) / cap;
    plan.per_launch = (NU + plan.launches - 1) / plan.launches;
  }
  return plan;
}
long chunks_per_unit(const FwdParams& p) {  // per sequence (the mean, with cu_seqlens)
  const long len = p.cu ? static_cast<long>(p.T) / std::max(p.num_seqs, 1) : static_cast<long>(p.T);
  return (len + tc::C - 1) / tc::C;
}


// Resets the status word (and the split kernel's record flags) and launches.
cudaError_t launch_chunk_tc_fwd(const FwdParams& p, cudaStream_t stream) {
  const long tokens = p.cu ? static_cast<long>(p.T) : static_cast<long>(p.num_seqs) * p.T;
  tc::Maps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!tc::make_map(&maps.q32, p.q, tc::KD, p.H, tokens, 32) || !tc::make_map(&maps.k32, p.k, tc::KD, p.H, tokens, 32) ||
      !tc::make_map(&maps.v, p.v, tc::VD, p.HV, tokens))
    return cudaErrorInvalidValue;
  const int NU = p.num_seqs * p.HV;
  const DeviceInfo& dev = device_info();
  const SplitPlan plan = split_plan(p.num_seqs, p.HV, chunks_per_unit(p), p.cu != nullptr);
  if (plan.launches > 0) {
    // one memset: the status word, the profile words and the flags behind them; a later
    // launch resets its flags only, so that the status word gathers every launch's reports
    if (cudaMemsetAsync(p.status, 0, kFlagOffset + plan.per_launch * kFlagBytesPerUnit, stream) != cudaSuccess)
      return cudaGetLastError();
    const int nt_max = (p.T + tc::C - 1) / tc::C;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(dev.sms);
    cfg.blockDim = dim3(tc::split::NTHREADS);
    cfg.dynamicSmemBytes = tc::split::SMEM_ALLOC;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!p.h && !tc::make_map(&maps.o, p.out, tc::VD, p.HV, tokens)) return cudaErrorInvalidValue;
    for (int b = 0; b < plan.launches; ++b) {
      FwdParams pb = p;
      pb.unit0 = b * plan.per_launch;
      const int nu = std::min(plan.per_launch, NU - pb.unit0);
      if (nu <= 0) break;
      if (b > 0 && cudaMemsetAsync(reinterpret_cast<uint8_t*>(p.status) + kFlagOffset, 0, nu * kFlagBytesPerUnit,
                                   stream) != cudaSuccess)
        return cudaGetLastError();
      const cudaError_t e = p.prestage
                                ? cudaLaunchKernelEx(&cfg, tc::kda_chunk_split_kernel<true>, maps, pb, nu, nt_max * nu)
                                : cudaLaunchKernelEx(&cfg, tc::kda_chunk_split_kernel<false>, maps, pb, nu, nt_max * nu);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream) != cudaSuccess) return cudaGetLastError();
  if (!dev.fused_attr) return cudaErrorInvalidConfiguration;
  dim3 grid(tc::NSLICE, p.HV, p.num_seqs);
  if (p.prestage)
    tc::kda_chunk_fused_kernel<true><<<grid, tc::NTHREADS, tc::SMEM_ALLOC, stream>>>(maps, p);
  else
    tc::kda_chunk_fused_kernel<false><<<grid, tc::NTHREADS, tc::SMEM_ALLOC, stream>>>(maps, p);
  return cudaGetLastError();
}

// Name of the kernel the chunked forward launches for this problem on the current device.
const char* chunk_kernel_name(bool bf16, int K, int V, long tokens, int num_seqs, int HV, bool packed) {
  const int units = num_seqs * HV;
  if (tokens <= 0 || units <= 0) return "none";
  if (!(bf16 && K == tc::KD && V == tc::VD && tc::encoder() != nullptr)) return "recurrent_fwd_kernel";
  const long len = tokens / num_seqs;
  return split_plan(num_seqs, HV, (len + tc::C - 1) / tc::C, packed).launches > 0 ? "kda_chunk_split_kernel"
                                                                                 : "kda_chunk_fused_kernel";
}

// Launches of that kernel per call (the split kernel covers many units in several).
int chunk_kernel_launches(bool bf16, int K, int V, long tokens, int num_seqs, int HV, bool packed) {
  const int units = num_seqs * HV;
  if (tokens <= 0 || units <= 0) return 0;
  if (!(bf16 && K == tc::KD && V == tc::VD && tc::encoder() != nullptr)) return 1;
  const long len = tokens / num_seqs;
  const SplitPlan plan = split_plan(num_seqs, HV, (len + tc::C - 1) / tc::C, packed);
  return plan.launches > 0 ? plan.launches : 1;
}

}  // namespace kda
