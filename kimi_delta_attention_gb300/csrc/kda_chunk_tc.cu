// kda_chunk_tc.cu -- fused tensor-core chunked KDA forward for sm_103a (bf16 I/O,
// K = V = 128, chunk C = 64).
//
// Chunked evaluation (page "手撕KDA", section "1 Naive", naive_chunk_kda; the
// decayed-operand factorisation follows the FlashKDA walk-through, page
// "KDA源码剖析之FlashKDA（上）", parts 9-11):
//   gc      = inclusive cumsum of g over the chunk rows, g_last = gc[C-1]
//   kd      = k e^{gc},  ki = k e^{-gc},  kr = k e^{g_last - gc},  qd = scale q e^{gc}
//   M       = strict_tril(Diag(beta) kd ki^T)           (beta scales rows)
//   Aqk     = tril(qd ki^T)                              (diagonal kept)
//   A       = (I + M)^{-1} Diag(beta)                    (beta scales columns)
//   W = A kd,  U = A v
//   per chunk, serially:  v_new = U - W S;  o = qd S + Aqk v_new;
//                         S <- Diag(e^{g_last}) S + kr^T v_new
//
// One CTA per (sequence, value head, 32-column slice of V): grid (4, HV, NS).
// Warps 0-3 ("prepare") build chunk n+1's operands while warps 4-7 ("chain")
// run chunk n's state update; the per-chunk record (qd, W, kr^T, Aqk, U, e^{g_last})
// is double-buffered in shared memory.  All dense contractions are tcgen05.mma
// (bf16 operands in 128-byte-swizzled shared memory, fp32 accumulators in TMEM):
//   prepare: L = kd ki^T, Aqk = qd ki^T (M=64,N=64,K=128); [W | U] = A [kd^T ; v^T]^T (M=64,N=160,K=64)
//   chain:   X = W S, O = qd S (M=64,N=32,K=128); P = kr^T v_new (M=128,N=32,K=64);
//            O += Aqk v_new (M=64,N=32,K=64)
// The K x 32 fp32 state slice lives in the chain threads' registers (thread d
// holds row d); its bf16 copy S^T in shared memory is the MMA operand.
// q, k and the v slice arrive by TMA; g and beta by coalesced register loads
// one chunk ahead.  The 64 x 64 unit-lower-triangular inverse runs on CUDA
// cores in fp32 (16 x 16 diagonal blocks by forward substitution, then block
// rows).  Every mbarrier wait is bounded; on a timeout the CTA records
// kStatusTimeout, drains, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "sm103.cuh"

namespace kda {
namespace tc {

constexpr int C = 64;         // chunk rows
constexpr int KD = 128;       // key dim
constexpr int VD = 128;       // value dim
constexpr int VS = 32;        // value columns per CTA
constexpr int NSLICE = VD / VS;
constexpr int NTHREADS = 256;
constexpr int MB_LD = 68;     // padded row stride (floats) of the fp32 inverse buffer

// ---- shared memory map (offsets from a 1024-aligned base) ----
constexpr uint32_t SET_BYTES = 65536;
constexpr uint32_t OFF_QD = 0;          // [64 x 128] bf16 SW128 (raw q lands here)
constexpr uint32_t OFF_WM = 16384;      // [64 x 128] bf16 SW128
constexpr uint32_t OFF_KRT = 32768;     // [128 x 64] bf16 SW128 (kr transposed)
constexpr uint32_t OFF_AQK = 49152;     // [64 x 64]  bf16 SW128
constexpr uint32_t OFF_U = 57344;       // [64 x 32]  fp32 row-major
constexpr uint32_t OFF_KD = 2 * SET_BYTES;       // 131072 [64 x 128] bf16 SW128
constexpr uint32_t OFF_KI = OFF_KD + 16384;      // 147456 [64 x 128] bf16 SW128 (raw k lands here)
constexpr uint32_t OFF_WUB = OFF_KI + 16384;     // 163840 [160 x 64] bf16 SW128: kd^T rows, then v^T rows
constexpr uint32_t OFF_AMAT = OFF_WUB + 20480;   // 184320 [64 x 64] bf16 SW128 (also fp32 scratch)
constexpr uint32_t OFF_ST = OFF_AMAT + 8192;     // 192512 [32 x 128] bf16 SW128 (S^T)
constexpr uint32_t OFF_VNT = OFF_ST + 8192;      // 200704 [32 x 64] bf16 SW128 (v_new^T)
constexpr uint32_t OFF_VST = OFF_VNT + 4096;     // 204800 [64 x 32] bf16 (raw v slice, TMA)
constexpr uint32_t OFF_MB = OFF_VST + 4096;      // 208896 [64 x 68] fp32 (M, then T in place)
constexpr uint32_t OFF_GAM = OFF_MB + 64 * MB_LD * 4;  // 226304 [2][128] fp32 e^{g_last}
constexpr uint32_t OFF_BETA = OFF_GAM + 1024;          // 227328 [64] fp32
constexpr uint32_t OFF_BAR = OFF_BETA + 256;           // 227584 mbarriers
constexpr uint32_t OFF_MISC = OFF_BAR + 128;           // 227712 tmem base, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;     // + alignment slack

// barrier slots
constexpr int BAR_RAW = 0, BAR_PMMA = 1, BAR_READY0 = 2, BAR_FREE0 = 4, BAR_A = 6, BAR_B = 7;

// TMEM columns
constexpr uint32_t TM_L = 0, TM_AQ = 64, TM_WU = 0, TM_X = 256, TM_O0 = 288, TM_P = 352;
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t RAW_TX_BYTES = 16384 + 16384 + 4096;  // q + k + v slice
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;        // 2 s

// named barriers
constexpr uint32_t NB_PREP = 1, NB_CHAIN = 2;

struct Maps {
  CUtensorMap q, k, v;
};

// Optional per-phase cycle counters (build with -DKDA_PROFILE): thread 0 of the
// prepare and chain warpgroups of block (0,0,0) accumulate clock64 deltas and
// store them after the status word in the workspace (16 + 16 uint64 slots).
#ifdef KDA_PROFILE
#define PROF_DECL uint64_t prof_acc[16] = {0}; uint64_t prof_last = clock64(); \
  const bool prof_on = (blockIdx.x | blockIdx.y | blockIdx.z) == 0;
#define PROF(i) do { if (prof_on) { const uint64_t t_ = clock64(); prof_acc[i] += t_ - prof_last; prof_last = t_; } } while (0)
#define PROF_STORE(base) do { if (prof_on) { uint64_t* dst_ = reinterpret_cast<uint64_t*>(p.status) + 1 + (base); \
  for (int i_ = 0; i_ < 16; ++i_) dst_[i_] = prof_acc[i_]; } } while (0)
#else
#define PROF_DECL
#define PROF(i) do { } while (0)
#define PROF_STORE(base) do { } while (0)
#endif

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return static_cast<uint32_t>(f2bf(lo)) | (static_cast<uint32_t>(f2bf(hi)) << 16);
}
__device__ __forceinline__ void st_v4(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

__global__ void __launch_bounds__(NTHREADS, 1)
kda_chunk_fused_kernel(const __grid_constant__ Maps maps, const FwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  float* gam = reinterpret_cast<float*>(sm + OFF_GAM);
  float* beta_s = reinterpret_cast<float*>(sm + OFF_BETA);
  float* mb = reinterpret_cast<float*>(sm + OFF_MB);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = blockIdx.x, hv = blockIdx.y, seq = blockIdx.z;
  const int HV = p.HV;
  const int hk = hv / (HV / p.H);
  const int v0 = slice * VS;

  long tok0;
  int len;
  seq_range(p, seq, tok0, len);
  const int NT = (len + C - 1) / C;

  if (tid == 0) {
    mbar_init(&bars[BAR_RAW], 1);
    mbar_init(&bars[BAR_PMMA], 1);
    mbar_init(&bars[BAR_READY0], 1);
    mbar_init(&bars[BAR_READY0 + 1], 1);
    mbar_init(&bars[BAR_FREE0], 1);
    mbar_init(&bars[BAR_FREE0 + 1], 1);
    mbar_init(&bars[BAR_A], 1);
    mbar_init(&bars[BAR_B], 1);
    fence_mbar_init();
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.k);
    tma_prefetch_desc(&maps.v);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const size_t state_off = (static_cast<size_t>(seq) * HV + hv) * KD * VD;

  if (warp < 4) {
    // =========================== prepare warpgroup ===========================
    const int pt = tid;  // key dim owned in the elementwise pass
    const int pw = warp;
    const float scale = p.scale;
    const float* gptr = p.g;
    uint32_t pmma_phase = 0;   // completed waits on the prepare MMA barrier
    uint32_t pmma_issued = 0;  // commits issued to it (elected thread)
    bool tma_pending = false;  // a raw load was issued and not yet waited for
    int pending_chunk = 0;
    bool failed = false;       // this thread saw a wait give up
    auto timeout = [&]() {
      failed = true;
      atomicOr(p.status, kStatusTimeout);
    };
    PROF_DECL

    auto issue_raw = [&](int n) {  // elected thread: TMA q, k, v slice of chunk n
      const int s = n & 1;
      const int row0 = static_cast<int>(tok0) + n * C;
      mbar_arrive_expect_tx(&bars[BAR_RAW], RAW_TX_BYTES);
      tma_load_3d(sm + s * SET_BYTES + OFF_QD, &maps.q, &bars[BAR_RAW], 0, hk, row0);
      tma_load_3d(sm + s * SET_BYTES + OFF_QD + 8192, &maps.q, &bars[BAR_RAW], 64, hk, row0);
      tma_load_3d(sm + OFF_KI, &maps.k, &bars[BAR_RAW], 0, hk, row0);
      tma_load_3d(sm + OFF_KI + 8192, &maps.k, &bars[BAR_RAW], 64, hk, row0);
      tma_load_3d(sm + OFF_VST, &maps.v, &bars[BAR_RAW], v0, hv, row0);
    };
    float gpre[C];
    float bpre = 0.f;
    auto prefetch_gb = [&](int n) {
      const int rows = min(C, len - n * C);
      const long base = tok0 + static_cast<long>(n) * C;
#pragma unroll
      for (int c = 0; c < C; ++c)
        gpre[c] = (c < rows) ? __ldg(gptr + (static_cast<size_t>(base + c) * HV + hv) * KD + pt) : 0.f;
      if (pt < C) bpre = (pt < rows) ? __ldg(p.beta + static_cast<size_t>(base + pt) * HV + hv) : 0.f;
    };

    if (NT > 0) {
      if (pt == 0) {
        issue_raw(0);
        tma_pending = true;
        pending_chunk = 0;
      }
      prefetch_gb(0);
    }

    for (int n = 0; n < NT; ++n) {
      const int s = n & 1;
      uint8_t* set = sm + s * SET_BYTES;
      const int rows = min(C, len - n * C);
      // ---- 1. raw q, k, v of chunk n ----
      if (!mbar_wait(&bars[BAR_RAW], n & 1, WAIT_LIMIT_NS)) timeout();
      if (named_bar_any(NB_PREP, 128, failed)) break;
      if (pt == 0) tma_pending = false;
      PROF(0);

      // ---- 2. elementwise: cumsum, decayed operands ----
      if (pt < C) beta_s[pt] = bpre;
      float glast = 0.f;
#pragma unroll
      for (int c = 0; c < C; ++c) glast += gpre[c];
      const float gamma = __expf(glast);
      gam[s * KD + pt] = gamma;
      {
        float gc = 0.f;
        uint8_t* qd_t = set + OFF_QD;
        uint8_t* ki_t = sm + OFF_KI;
        uint8_t* kd_t = sm + OFF_KD;
#pragma unroll
        for (int c8 = 0; c8 < C / 8; ++c8) {
          uint32_t kdT[4], krT[4];
#pragma unroll
          for (int cc = 0; cc < 8; cc += 2) {
            float kdv[2], krv[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = c8 * 8 + cc + h;
              gc += gpre[c];
              const float e = __expf(gc);
              const float ie = __expf(-gc);
              const uint32_t off = sw128_offset(c, pt, C);
              const bool valid = c < rows;
              const float kv = valid ? bf2f(*reinterpret_cast<const uint16_t*>(ki_t + off)) : 0.f;
              const float qv = valid ? bf2f(*reinterpret_cast<const uint16_t*>(qd_t + off)) : 0.f;
              const float kdf = kv * e;
              const float kif = kv * ie;
              kdv[h] = kdf;
              krv[h] = kif * gamma;
              *reinterpret_cast<uint16_t*>(kd_t + off) = f2bf(kdf);
              *reinterpret_cast<uint16_t*>(ki_t + off) = f2bf(kif);
              *reinterpret_cast<uint16_t*>(qd_t + off) = f2bf(qv * e * scale);
            }
            kdT[cc / 2] = pack2(kdv[0], kdv[1]);
            krT[cc / 2] = pack2(krv[0], krv[1]);
          }
          st_v4(sm + OFF_WUB + sw128_offset(pt, c8 * 8, 160), kdT[0], kdT[1], kdT[2], kdT[3]);
          st_v4(set + OFF_KRT + sw128_offset(pt, c8 * 8, 128), krT[0], krT[1], krT[2], krT[3]);
        }
      }
      {  // v slice transposed into rows 128..159 of the W/U B operand
        const int vv = pt >> 2, cb = (pt & 3) * 16;
        const uint16_t* vst = reinterpret_cast<const uint16_t*>(sm + OFF_VST);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const int c = cb + h * 8 + i;
            const float a = (c < rows) ? bf2f(vst[c * VS + vv]) : 0.f;
            const float b = (c + 1 < rows) ? bf2f(vst[(c + 1) * VS + vv]) : 0.f;
            w[i / 2] = pack2(a, b);
          }
          st_v4(sm + OFF_WUB + sw128_offset(128 + vv, cb + h * 8, 160), w[0], w[1], w[2], w[3]);
        }
      }
      if (n + 1 < NT) prefetch_gb(n + 1);
      fence_proxy_async_smem();
      named_bar_sync(NB_PREP, 128);
      PROF(1);

      // ---- 3. L = kd ki^T, Aqk = qd ki^T ----
      if (pt == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_f16kind(64, 64);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t koff = kb * 8192 + ks * 32;
            const uint64_t bd = sdesc_sw128(smem_u32(sm + OFF_KI + koff));
            umma_f16(tmem + TM_L, sdesc_sw128(smem_u32(sm + OFF_KD + koff)), bd, idesc, (kb | ks) != 0);
            umma_f16(tmem + TM_AQ, sdesc_sw128(smem_u32(set + OFF_QD + koff)), bd, idesc, (kb | ks) != 0);
          }
        umma_commit(&bars[BAR_PMMA]);
        ++pmma_issued;
      }
      __syncwarp();
      if (!mbar_wait(&bars[BAR_PMMA], pmma_phase & 1, WAIT_LIMIT_NS)) timeout();
      ++pmma_phase;
      tc_fence_after();
      PROF(2);

      // KI and VST are free again: fetch chunk n+1 (its set must be released by the chain)
      if (pt == 0 && n + 1 < NT && !failed) {
        bool ok = true;
        if (n + 1 >= 2) ok = mbar_wait(&bars[BAR_FREE0 + ((n + 1) & 1)], ((n - 1) >> 1) & 1, WAIT_LIMIT_NS);
        if (ok) {
          issue_raw(n + 1);
          tma_pending = true;
          pending_chunk = n + 1;
        } else {
          timeout();
        }
      }
      PROF(3);

      // ---- 4. TMEM -> M (fp32, rows scaled by beta, strictly lower) and Aqk (bf16, lower) ----
      __syncwarp();
      {
        const int i = 16 * pw + (lane & 15);
        float r[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld32(tmem_addr(tmem, 32 * pw, TM_L + 32 * half), r);
          tmem_ld_wait();
          if (lane < 16) {
            const float bi = beta_s[i];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              float4 v4;
              const int j = 32 * half + 4 * j4;
              v4.x = (j + 0 < i) ? bi * r[4 * j4 + 0] : 0.f;
              v4.y = (j + 1 < i) ? bi * r[4 * j4 + 1] : 0.f;
              v4.z = (j + 2 < i) ? bi * r[4 * j4 + 2] : 0.f;
              v4.w = (j + 3 < i) ? bi * r[4 * j4 + 3] : 0.f;
              *reinterpret_cast<float4*>(mb + i * MB_LD + j) = v4;
            }
          }
          tmem_ld32(tmem_addr(tmem, 32 * pw, TM_AQ + 32 * half), r);
          tmem_ld_wait();
          if (lane < 16) {
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int j = 32 * half + 8 * j8 + 2 * t;
                w[t] = pack2((j <= i) ? r[8 * j8 + 2 * t] : 0.f, (j + 1 <= i) ? r[8 * j8 + 2 * t + 1] : 0.f);
              }
              st_v4(set + OFF_AQK + sw128_offset(i, 32 * half + 8 * j8, 64), w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      tc_fence_before();
      if (named_bar_any(NB_PREP, 128, failed)) break;
      PROF(4);

      // ---- 5. T = (I + M)^{-1}: 16x16 diagonal blocks, then block rows ----
      {
        if (lane < 16) {
          const int b0 = 16 * pw, j = lane;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m) acc = fmaf(-mb[(b0 + i) * MB_LD + b0 + m], x[m], acc);
            x[i] = acc;
          }
          __syncwarp(0x0000FFFFu);
#pragma unroll
          for (int i = 0; i < 16; ++i) mb[(b0 + i) * MB_LD + b0 + j] = x[i];
        }
        named_bar_sync(NB_PREP, 128);
        PROF(5);
        float* rs = reinterpret_cast<float*>(sm + OFF_AMAT);  // [16][48] fp32 scratch
        const int r = pt >> 3;
        for (int bi = 1; bi < 4; ++bi) {
          const int ncol = 16 * bi;          // columns of the block row left of the diagonal
          const int per = 2 * bi;            // elements per thread
          const int c0 = (pt & 7) * per;
          const float* mrow = mb + (16 * bi + r) * MB_LD;
          for (int e = 0; e < per; ++e) {    // R = M_i[:, :16i] T[:16i, :16i]
            const int c = c0 + e;
            float acc = 0.f;
            for (int k = c; k < ncol; ++k) acc = fmaf(mrow[k], mb[k * MB_LD + c], acc);
            rs[r * 48 + c] = acc;
          }
          named_bar_sync(NB_PREP, 128);
          const float* trow = mb + (16 * bi + r) * MB_LD + 16 * bi;  // T_ii row r
          for (int e = 0; e < per; ++e) {    // T_i[:, :16i] = -T_ii R
            const int c = c0 + e;
            float acc = 0.f;
            for (int m = 0; m <= r; ++m) acc = fmaf(trow[m], rs[m * 48 + c], acc);
            mb[(16 * bi + r) * MB_LD + c] = -acc;
          }
          named_bar_sync(NB_PREP, 128);
        }
        PROF(6);
        // A = T Diag(beta) -> bf16 SW128
        {
          const int i = pt >> 1, jb = (pt & 1) * 32;
#pragma unroll
          for (int j8 = 0; j8 < 4; ++j8) {
            uint32_t w[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int j = jb + 8 * j8 + 2 * t;
              const float a = (j <= i) ? mb[i * MB_LD + j] * beta_s[j] : 0.f;
              const float b = (j + 1 <= i) ? mb[i * MB_LD + j + 1] * beta_s[j + 1] : 0.f;
              w[t] = pack2(a, b);
            }
            st_v4(sm + OFF_AMAT + sw128_offset(i, jb + 8 * j8, 64), w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(NB_PREP, 128);
      PROF(7);

      // ---- 6. [W | U] = A [kd^T ; v^T]^T ----
      if (pt == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_f16kind(64, 160);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16(tmem + TM_WU, sdesc_sw128(smem_u32(sm + OFF_AMAT + ks * 32)),
                   sdesc_sw128(smem_u32(sm + OFF_WUB + ks * 32)), idesc, ks != 0);
        umma_commit(&bars[BAR_PMMA]);
        ++pmma_issued;
      }
      __syncwarp();
      if (!mbar_wait(&bars[BAR_PMMA], pmma_phase & 1, WAIT_LIMIT_NS)) timeout();
      ++pmma_phase;
      tc_fence_after();
      PROF(8);

      // ---- 7. W -> bf16 SW128, U -> fp32 ----
      __syncwarp();
      {
        const int i = 16 * pw + (lane & 15);
        float r[32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          tmem_ld32(tmem_addr(tmem, 32 * pw, TM_WU + 32 * q4), r);
          tmem_ld_wait();
          if (lane < 16) {
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8)
              st_v4(set + OFF_WM + sw128_offset(i, 32 * q4 + 8 * j8, 64), pack2(r[8 * j8], r[8 * j8 + 1]),
                    pack2(r[8 * j8 + 2], r[8 * j8 + 3]), pack2(r[8 * j8 + 4], r[8 * j8 + 5]),
                    pack2(r[8 * j8 + 6], r[8 * j8 + 7]));
          }
        }
        tmem_ld32(tmem_addr(tmem, 32 * pw, TM_WU + 128), r);
        tmem_ld_wait();
        if (lane < 16) {
          float4* urow = reinterpret_cast<float4*>(set + OFF_U + i * (VS * 4));
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) urow[j4] = make_float4(r[4 * j4], r[4 * j4 + 1], r[4 * j4 + 2], r[4 * j4 + 3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      if (named_bar_any(NB_PREP, 128, failed)) break;
      if (pt == 0) mbar_arrive(&bars[BAR_READY0 + s]);
      PROF(9);
    }
    // drain after an abort: copies and MMAs still in flight must finish before
    // the CTA frees TMEM and exits
    if (pt == 0) {
      if (tma_pending && !mbar_wait(&bars[BAR_RAW], pending_chunk & 1, WAIT_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
      if (pmma_issued > pmma_phase && !mbar_wait(&bars[BAR_PMMA], (pmma_issued - 1) & 1, WAIT_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
      PROF_STORE(0);
    }
  } else {
    // ============================= chain warpgroup =============================
    const int qt = tid - 128;   // state row d
    const int qw = warp - 4;    // TMEM lane quadrant
    const int d = qt;
    float st[VS];
    if (p.s0) {
      const float4* src = reinterpret_cast<const float4*>(p.s0 + state_off + static_cast<size_t>(d) * VD + v0);
#pragma unroll
      for (int j4 = 0; j4 < VS / 4; ++j4) {
        const float4 v4 = src[j4];
        st[4 * j4] = v4.x; st[4 * j4 + 1] = v4.y; st[4 * j4 + 2] = v4.z; st[4 * j4 + 3] = v4.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < VS; ++j) st[j] = 0.f;
    }
    auto write_st = [&]() {
#pragma unroll
      for (int j = 0; j < VS; ++j)
        *reinterpret_cast<uint16_t*>(sm + OFF_ST + sw128_offset(j, d, VS)) = f2bf(st[j]);
    };
    write_st();
    fence_proxy_async_smem();
    named_bar_sync(NB_CHAIN, 128);

    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    bool failed = false;
    bool aborted = false;
    int a_issued = 0, b_issued = 0, a_done = 0, b_done = 0;  // commits (elected thread) / waits
    auto timeout = [&]() {
      failed = true;
      atomicOr(p.status, kStatusTimeout);
    };
    PROF_DECL
    for (int n = 0; n < NT; ++n) {
      const int s = n & 1;
      uint8_t* set = sm + s * SET_BYTES;
      const int rows = min(C, len - n * C);
      // ---- X = W S, O = qd S ----
      if (qt == 0) {
        if (!mbar_wait(&bars[BAR_READY0 + s], (n >> 1) & 1, WAIT_LIMIT_NS)) {
          timeout();
        } else {
          tc_fence_after();
          constexpr uint32_t idesc = idesc_f16kind(64, VS);
#pragma unroll
          for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bd = sdesc_sw128(smem_u32(sm + OFF_ST + kb * 4096 + ks * 32));
              const uint32_t koff = kb * 8192 + ks * 32;
              umma_f16(tmem + TM_X, sdesc_sw128(smem_u32(set + OFF_WM + koff)), bd, idesc, (kb | ks) != 0);
              umma_f16(tmem + TM_O0 + 32 * s, sdesc_sw128(smem_u32(set + OFF_QD + koff)), bd, idesc,
                       (kb | ks) != 0);
            }
          umma_commit(&bars[BAR_A]);
          ++a_issued;
        }
      }
      PROF(0);
      __syncwarp();
      if (!mbar_wait(&bars[BAR_A], n & 1, WAIT_LIMIT_NS)) timeout();
      ++a_done;
      tc_fence_after();
      PROF(1);
      // ---- v_new = U - X  ->  v_new^T (bf16 SW128) ----
      {
        float xr[32];
        tmem_ld32(tmem_addr(tmem, 32 * qw, TM_X), xr);
        tmem_ld_wait();
        if (lane < 16) {
          const int c = 16 * qw + lane;
          const float4* urow = reinterpret_cast<const float4*>(set + OFF_U + c * (VS * 4));
#pragma unroll
          for (int j4 = 0; j4 < VS / 4; ++j4) {
            const float4 u4 = urow[j4];
            const float vn[4] = {u4.x - xr[4 * j4], u4.y - xr[4 * j4 + 1], u4.z - xr[4 * j4 + 2],
                                 u4.w - xr[4 * j4 + 3]};
#pragma unroll
            for (int t = 0; t < 4; ++t)
              *reinterpret_cast<uint16_t*>(sm + OFF_VNT + sw128_offset(4 * j4 + t, c, VS)) = f2bf(vn[t]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (named_bar_any(NB_CHAIN, 128, failed)) {
        aborted = true;
        break;
      }
      PROF(2);
      // ---- P = kr^T v_new ; O += Aqk v_new ----
      if (qt == 0) {
        tc_fence_after();
        constexpr uint32_t idesc_p = idesc_f16kind(128, VS);
        constexpr uint32_t idesc_o = idesc_f16kind(64, VS);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = sdesc_sw128(smem_u32(sm + OFF_VNT + ks * 32));
          umma_f16(tmem + TM_P, sdesc_sw128(smem_u32(set + OFF_KRT + ks * 32)), bd, idesc_p, ks != 0);
          umma_f16(tmem + TM_O0 + 32 * s, sdesc_sw128(smem_u32(set + OFF_AQK + ks * 32)), bd, idesc_o, 1u);
        }
        umma_commit(&bars[BAR_B]);
        ++b_issued;
      }
      __syncwarp();
      if (!mbar_wait(&bars[BAR_B], n & 1, WAIT_LIMIT_NS)) timeout();
      ++b_done;
      tc_fence_after();
      PROF(3);
      // ---- S <- Diag(e^{g_last}) S + P ; refresh S^T ----
      __syncwarp();
      {
        float pr[32];
        tmem_ld32(tmem_addr(tmem, 32 * qw, TM_P), pr);
        tmem_ld_wait();
        const float gmm = gam[s * KD + d];
#pragma unroll
        for (int j = 0; j < VS; ++j) st[j] = fmaf(gmm, st[j], pr[j]);
        write_st();
      }
      PROF(4);
      // ---- o rows of this chunk ----
      {
        float orr[32];
        tmem_ld32(tmem_addr(tmem, 32 * qw, TM_O0 + 32 * s), orr);
        tmem_ld_wait();
        const int c = 16 * qw + lane;
        if (lane < 16 && c < rows) {
          uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(tok0 + n * C + c) * HV + hv) * VD + v0);
#pragma unroll
          for (int j8 = 0; j8 < VS / 8; ++j8)
            dst[j8] = make_uint4(pack2(orr[8 * j8], orr[8 * j8 + 1]), pack2(orr[8 * j8 + 2], orr[8 * j8 + 3]),
                                 pack2(orr[8 * j8 + 4], orr[8 * j8 + 5]), pack2(orr[8 * j8 + 6], orr[8 * j8 + 7]));
        }
      }
      PROF(5);
      fence_proxy_async_smem();
      tc_fence_before();
      if (named_bar_any(NB_CHAIN, 128, failed)) {
        aborted = true;
        break;
      }
      if (qt == 0) mbar_arrive(&bars[BAR_FREE0 + s]);
      PROF(6);
    }
    if (qt == 0) {  // drain MMAs still in flight after an abort
      if (a_issued > a_done && !mbar_wait(&bars[BAR_A], (a_issued - 1) & 1, WAIT_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
      if (b_issued > b_done && !mbar_wait(&bars[BAR_B], (b_issued - 1) & 1, WAIT_LIMIT_NS))
        atomicOr(p.status, kStatusTimeout);
      PROF_STORE(16);
    }
    if (p.sfin && !aborted) {
      float4* dst = reinterpret_cast<float4*>(p.sfin + state_off + static_cast<size_t>(d) * VD + v0);
#pragma unroll
      for (int j4 = 0; j4 < VS / 4; ++j4)
        dst[j4] = make_float4(st[4 * j4], st[4 * j4 + 1], st[4 * j4 + 2], st[4 * j4 + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
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

// 3-D map over a [tokens, heads, dim] bf16 tensor with a (box_x, 1, 64) box.
bool make_map(CUtensorMap* m, const void* base, int dim, int heads, long tokens, int box_x, bool swizzle) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dim) * 2, static_cast<cuuint64_t>(heads) * dim * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_x), 1, static_cast<cuuint32_t>(C)};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

bool chunk_tc_supported(const FwdParams& p, bool bf16) {
  const long tokens = p.cu ? static_cast<long>(p.T) : static_cast<long>(p.num_seqs) * p.T;
  return bf16 && p.K == tc::KD && p.V == tc::VD && tokens > 0 && tc::encoder() != nullptr;
}

cudaError_t launch_chunk_tc_fwd(const FwdParams& p, cudaStream_t stream) {
  const long tokens = p.cu ? static_cast<long>(p.T) : static_cast<long>(p.num_seqs) * p.T;
  tc::Maps maps;
  if (!tc::make_map(&maps.q, p.q, tc::KD, p.H, tokens, 64, true) ||
      !tc::make_map(&maps.k, p.k, tc::KD, p.H, tokens, 64, true) ||
      !tc::make_map(&maps.v, p.v, tc::VD, p.HV, tokens, tc::VS, false))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc::kda_chunk_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tc::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(tc::NSLICE, p.HV, p.num_seqs);
  tc::kda_chunk_fused_kernel<<<grid, tc::NTHREADS, tc::SMEM_ALLOC, stream>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace kda
