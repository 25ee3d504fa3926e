// kda_backward_chunk.cu -- the backward in chunk form: gradients of
// sum_t <do_t, o_t> + <dS_final, S_final> with respect to q, k, v, g, beta and the
// initial state, chunk by chunk (C = 64), with every contraction on the tensor cores and
// each operand split into a high and a low part, so that three products give fp32-level
// accuracy: tcgen05 products of bf16 parts (accumulators in TMEM) for the state chains,
// the value-side gradients and the preparation's K x K / K x V products when K = V = 128;
// warp-level m16n8k8 products of TF32 parts for the rest and for other head sizes.
//
// The forward of a chunk (page "手撕KDA", section "1 Naive": the chunked form; gc the
// cumulative sum of g inside the chunk, gl its last row, S the state entering it):
//     kd = k e^{gc}, ki = k e^{-gc}, qd = scale q e^{gc}, kr = k e^{gl - gc}
//     M = strict_tril(Diag(beta) kd ki^T), T = (I + M)^{-1}, A = T Diag(beta)
//     W = A kd, U = A v, v_new = U - W S, Aqk = tril(qd ki^T)
//     o = qd S + Aqk v_new,   S' = Diag(e^{gl}) S + kr^T v_new.
// So S' = Q S + R with Q = Diag(e^{gl}) - kr^T W and R = kr^T U, and going back,
//     dv_new = Aqk^T do + kr dS',   dS = Q^T dS' + B,   B = qd^T do - W^T Aqk^T do,
// and the section "2 Backward" chain rule through the chunk's products:
//     dAqk = tril(do v_new^T), dW = -dv_new S^T, dA = dW kd^T + dv_new v^T,
//     dv = A^T dv_new, dkd = A^T dW, dbeta_j += sum_i T_ij dA_ij,
//     dM = -strict_tril(T^T dA A^T), dbeta_i += sum_j dM_ij (kd ki^T)_ij,
//     dq = scale e^{gc} (do S^T + dAqk ki),  dk = e^{gc} (dkd + dMb ki) + e^{-gc} (dAqk^T qd + dMb^T kd)
//          + e^{gl - gc} (v_new dS'^T),   dMb = Diag(beta) dM,
//     dgc = q dq + k (dk_e^{gc} - dk_e^{-gc} - dk_e^{gl-gc}),  dgl += e^{gl} sum_v S dS' + sum_i k dk_e^{gl-gc},
//     dg = the reverse cumulative sum of dgc (dgl added at the chunk's last row).
//
// Range.  The factors e^{gc_i - gc_j} of the products over a chunk's rows are formed
// block by block (16-row blocks b with reference points s_b, e_b: gc just before and at
// the end of the block), each factor between 0 and e^{-(decay of one block)}, the
// limit the forward kernels also have; e^{gc}, e^{gl - gc} never exceed 1.
//
// Five launches, each parallel over (chunk, value head) except the chains:
//   prep_kernel       Q, R, B of every chunk, and W, U, Aqk^T do, T and kd ki^T for the
//                     gradient kernels (workspace slot per (chunk, value head));
//   chain_tc_kernel   the states entering each chunk (h_{n+1} = Q_n h_n + R_n) and the
//   (chain_kernel)    state gradients leaving it (dS_n = Q_n^T dS_{n+1} + B_n), one CTA per
//                     64 value columns and direction (the columns are independent);
//   grad_v_tc_kernel  v_new, dv_new and the products with S and dS' (dv final);
//   (grad_v_kernel)
//   grad_cc_kernel    dA, dM and dbeta (C x C);
//   grad_k_kernel     dq, dk, dg (per 64 key dims).
// (the kernels in parentheses: K = 64 or V = 64)
#include "kda_common.cuh"
#include "sm103.cuh"

namespace kda {
namespace cbwd {

constexpr int NT = 256, NW = 8, C = 64;  // 16-row blocks inside a chunk
constexpr int LC = C + 4;  // padded row of a C x C fp32 tile (row stride = 4 mod 32 banks)
constexpr float kLog2e = 1.4426950408889634f;
#ifndef KDA_CBWD_SPLIT
#define KDA_CBWD_SPLIT 1
#endif
constexpr bool kSplit = KDA_CBWD_SPLIT != 0;
// The decay of one 16-row block that the block factors hold (log2 units, as the forward
// kernels): beyond it a chunk raises the status range bit.
constexpr float kMinBlockLog2 = -116.f;
// Waits for a CTA's own copies and products give up after Params::wait_ns (the status
// then reports a timeout); draining them before the CTA releases its memory always allows
// this much.
constexpr unsigned long long kDrainNs = 2000000000ull;

struct Params {
  const void* q;       // [tokens, H, K]  io type
  const void* k;
  const void* v;       // [tokens, HV, V]  io type
  const float* g;      // [tokens, HV, K]
  const float* beta;   // [tokens, HV]
  const float* s0;     // [NS, HV, K, V] or null
  const int32_t* cu;   // [NS + 1] or null
  const void* d_out;   // [tokens, HV, V]  io type
  const float* d_fin;  // [NS, HV, K, V] or null
  float* dq;           // [tokens, H, K]  accumulated (zeroed by the launcher)
  float* dk;
  float* dv;           // [tokens, HV, V]
  float* dg;           // [tokens, HV, K]
  float* dbeta;        // [tokens, HV]
  float* ds0;          // [NS, HV, K, V] or null
  float* ws;           // slots, one per (flat chunk, value head)
  uint32_t* status;
  size_t slot_floats;
  unsigned long long wait_ns;  // limit of a bounded wait (tcgen05 chains)
  float scale;
  int T, H, HV, num_seqs;
  int nc;              // chunks per sequence (fixed length)
};

// Per-slot layout (floats, dense rows): the chains' operands, then what the gradient
// kernels hand on.  RH holds R until the forward chain replaces it by the state
// entering the chunk, BD holds B until the reverse chain replaces it by dS'.
template <int K, int V>
struct Slot {
  static constexpr size_t Q = 0, RH = Q + K * K, BD = RH + K * V, W = BD + K * V, U = W + C * K, E = U + C * V,
                          T = E + C * V, KK = T + C * C, DH = KK + C * C, DW = DH + C * K, DKR = DW + C * K,
                          DAQK = DKR + C * K, DAV = DAQK + C * C, DMB = DAV + C * C, DGL = DMB + C * C,
                          FLOATS = DGL + K;
};

// Element (key row d, value column v) of the K x V regions RH and BD: 64-column slices
// stored one after the other (each K x 64, rows of 64), so that a chain CTA's slice is
// one contiguous block.
template <int K>
__device__ __forceinline__ size_t kv_off(int d, int v) {
  return static_cast<size_t>(v >> 6) * (K * 64) + static_cast<size_t>(d) * 64 + (v & 63);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}

// Flat chunk f (chunks numbered sequence by sequence) -> its sequence, chunk within the
// sequence, first token and rows; false past the last chunk or on a bad cu_seqlens.
__device__ bool find_chunk(const Params& p, int f, int& seq, int& m, long& tok0, int& rows) {
  if (!p.cu) {
    seq = f / p.nc;
    m = f - seq * p.nc;
    if (seq >= p.num_seqs) return false;
    tok0 = static_cast<long>(seq) * p.T + static_cast<long>(m) * C;
    rows = min(C, p.T - m * C);
    return true;
  }
  int f0 = 0;
  for (int s = 0; s < p.num_seqs; ++s) {
    const int a = p.cu[s], b = p.cu[s + 1];
    if (a < 0 || b < a || b > p.T || (s == 0 && a != 0) || (s == p.num_seqs - 1 && b != p.T)) {
      atomicOr(p.status, kStatusBounds);
      return false;
    }
    const int n = (b - a + C - 1) / C;
    if (f < f0 + n) {
      seq = s;
      m = f - f0;
      tok0 = a + static_cast<long>(m) * C;
      rows = min(C, b - a - m * C);
      return true;
    }
    f0 += n;
  }
  return false;
}
// First flat chunk and chunk count of sequence `seq`.
__device__ bool seq_chunks(const Params& p, int seq, int& f0, int& nch) {
  if (!p.cu) {
    f0 = seq * p.nc;
    nch = p.nc;
    return true;
  }
  f0 = 0;
  for (int s = 0; s <= seq; ++s) {
    const int a = p.cu[s], b = p.cu[s + 1];
    if (a < 0 || b < a || b > p.T || (s == 0 && a != 0) || (s == p.num_seqs - 1 && b != p.T)) {
      atomicOr(p.status, kStatusBounds);
      return false;
    }
    nch = (b - a + C - 1) / C;
    if (s < seq) f0 += nch;
  }
  return true;
}

// C rows of N columns (io type) into fp32 shared memory with row stride N + 4; rows
// past `rows` are zero.
// (all of a thread's loads are issued before its stores: C N / 4 is a multiple of NT)
template <typename IO, int N>
__device__ __forceinline__ void load_rows(float* dst, const IO* src, long row0, int rows, size_t row_stride,
                                          size_t col0) {
  constexpr int PER = C * (N / 4) / NT;
  static_assert(C * (N / 4) % NT == 0, "whole passes");
  float4 x[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int idx = threadIdx.x + u * NT, r = idx / (N / 4), c4 = (idx - r * (N / 4)) * 4;
    x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < rows) x[u] = load4(src + static_cast<size_t>(row0 + r) * row_stride + col0 + c4);
  }
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int idx = threadIdx.x + u * NT, r = idx / (N / 4), c4 = (idx - r * (N / 4)) * 4;
    *reinterpret_cast<float4*>(dst + r * (N + 4) + c4) = x[u];
  }
}
// rows x N dense fp32 (global) <-> shared memory with row stride LD
template <int N, int LD>
__device__ __forceinline__ void copy_in(float* dst, const float* src) {
  constexpr int PER = C * (N / 4) / NT;
  static_assert(C * (N / 4) % NT == 0, "whole passes");
  float4 x[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int idx = threadIdx.x + u * NT, r = idx / (N / 4), c4 = (idx - r * (N / 4)) * 4;
    x[u] = load4(src + static_cast<size_t>(r) * N + c4);
  }
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int idx = threadIdx.x + u * NT, r = idx / (N / 4), c4 = (idx - r * (N / 4)) * 4;
    *reinterpret_cast<float4*>(dst + r * LD + c4) = x[u];
  }
}
template <int N, int LD>
__device__ __forceinline__ void copy_out(float* dst, const float* src) {
  for (int idx = threadIdx.x; idx < C * (N / 4); idx += NT) {
    const int r = idx / (N / 4), c4 = (idx - r * (N / 4)) * 4;
    *reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * N + c4) = *reinterpret_cast<const float4*>(src + r * LD + c4);
  }
}

// In-place cumulative sum down the C rows of columns [0, N) (stride LD), in log2 units.
template <int N, int LD>
__device__ __forceinline__ void cumsum_log2(float* x) {
  for (int d = threadIdx.x; d < N; d += NT) {
    float s = 0.f;
#pragma unroll 16
    for (int i = 0; i < C; ++i) {
      s = fmaf(x[i * LD + d], kLog2e, s);
      x[i * LD + d] = s;
    }
  }
}

// ------------------------------------------------------------ warp products --
// One warp accumulates MT stacked 16 x (8 NT8) tiles at (m0 + 16 mt, n0) of
// sum_k A(m, k) B(k, n) over k in [kb, ke) (multiples of 8).  fa(m, k, n0) and
// fb(k, n, m0) return fp32 operands; each is split into TF32 high and low parts and the
// three products lo*hi, hi*lo, hi*hi accumulate in fp32 (kSplit), else a single TF32
// product.  The fragments of a k-step are loaded first, then the products run in passes
// over all accumulators, so that no product waits on the one before it.
template <int MT, int NT8, class FA, class FB>
__device__ __forceinline__ void kstep_mma(float (&a0)[MT][NT8][4], float (&a1)[MT][NT8][4], float (&a2)[MT][NT8][4],
                                          const FA& fa, const FB& fb, int m0, int n0, int k) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  uint32_t ah[MT][4], al[MT][4], bh[NT8][2], bl[NT8][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int m = m0 + 16 * mt + g;
    const float av[4] = {fa(m, k + t, n0), fa(m + 8, k + t, n0), fa(m, k + t + 4, n0), fa(m + 8, k + t + 4, n0)};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ah[mt][e] = to_tf32(av[e]);
      if (kSplit) al[mt][e] = to_tf32(av[e] - __uint_as_float(ah[mt][e]));
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT8; ++nt) {
    const int n = n0 + 8 * nt + g;
    const float bv[2] = {fb(k + t, n, m0), fb(k + t + 4, n, m0)};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      bh[nt][e] = to_tf32(bv[e]);
      if (kSplit) bl[nt][e] = to_tf32(bv[e] - __uint_as_float(bh[nt][e]));
    }
  }
  if (kSplit) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt) mma_tf32_m16n8k8(a1[mt][nt], al[mt], bh[nt][0], bh[nt][1]);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt) mma_tf32_m16n8k8(a2[mt][nt], ah[mt], bl[nt][0], bl[nt][1]);
  }
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) mma_tf32_m16n8k8(a0[mt][nt], ah[mt], bh[nt][0], bh[nt][1]);
}
// One warp accumulates MT stacked 16 x (8 NT8) tiles at (m0 + 16 mt, n0) of
// sum_k A(m, k) B(k, n) over k in [kb, ke) (multiples of 8).  fa(m, k, n0) and
// fb(k, n, m0) return fp32 operands; each is split into TF32 high and low parts and the
// three products lo*hi, hi*lo, hi*hi accumulate in fp32 (kSplit), else a single TF32
// product.  The fragments of a k-step are loaded first, then the products run in passes
// over all accumulators, so that no product waits on the one before it; tiles with at
// most two accumulators spread the three products and alternate k-steps over six
// partial sums (added at the end), which keeps as many products independent.
template <int MT, int NT8, class FA, class FB>
__device__ __forceinline__ void tile_mma(float (&acc)[MT][NT8][4], const FA& fa, const FB& fb, int m0, int n0, int kb,
                                         int ke) {
  if constexpr (MT * NT8 <= 2) {
    float p[5][MT][NT8][4];
#pragma unroll
    for (int i = 0; i < 5; ++i)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) p[i][mt][nt][e] = 0.f;
    int k = kb;
    for (; k + 16 <= ke; k += 16) {
      kstep_mma<MT, NT8>(acc, p[0], p[1], fa, fb, m0, n0, k);
      kstep_mma<MT, NT8>(p[2], p[3], p[4], fa, fb, m0, n0, k + 8);
    }
    if (k < ke) kstep_mma<MT, NT8>(acc, p[0], p[1], fa, fb, m0, n0, k);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          acc[mt][nt][e] += ((p[0][mt][nt][e] + p[1][mt][nt][e]) + (p[2][mt][nt][e] + p[3][mt][nt][e])) + p[4][mt][nt][e];
  } else {
#pragma unroll 2
    for (int k = kb; k < ke; k += 8) kstep_mma<MT, NT8>(acc, acc, acc, fa, fb, m0, n0, k);
  }
}
// single 16-row tile
template <int NT8, class FA, class FB>
__device__ __forceinline__ void tile_mma(float (&acc)[NT8][4], const FA& fa, const FB& fb, int m0, int n0, int kb,
                                         int ke) {
  tile_mma<1, NT8>(reinterpret_cast<float(&)[1][NT8][4]>(acc), fa, fb, m0, n0, kb, ke);
}
// accumulator element e of n-tile nt: row m0 + g + 8 (e >> 1), column n0 + 8 nt + 2 t + (e & 1)
template <int NT8, class FI>
__device__ __forceinline__ void tile_init(float (&acc)[NT8][4], const FI& init, int m0, int n0) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = init(m0 + g + 8 * (e >> 1), n0 + 8 * nt + 2 * t + (e & 1));
}
template <int NT8, class FE>
__device__ __forceinline__ void tile_epi(const float (&acc)[NT8][4], const FE& epi, int m0, int n0) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT8; ++nt) {
    epi(m0 + g, n0 + 8 * nt + 2 * t, acc[nt][0], acc[nt][1]);
    epi(m0 + g + 8, n0 + 8 * nt + 2 * t, acc[nt][2], acc[nt][3]);
  }
}
// The whole M x N product over the CTA's warps, tile by tile (MT x 16 rows by 8 NT8
// columns): init, the k range krange(m0, n0) (int2), epilogue on column pairs.  Tiles for
// which live(m0, n0) is false keep their init values.
template <int M, int N, int NT8, int MT, class FA, class FB, class FL, class FR, class FI, class FE>
__device__ __forceinline__ void cta_gemm(const FA& fa, const FB& fb, const FL& live, const FR& krange, const FI& init,
                                         const FE& epi) {
  constexpr int TN = N / (8 * NT8), TILES = (M / (16 * MT)) * TN;
  const int warp = threadIdx.x >> 5;
  for (int tile = warp; tile < TILES; tile += NW) {
    const int m0 = (tile / TN) * 16 * MT, n0 = (tile % TN) * (8 * NT8);
    float acc[MT][NT8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) tile_init<NT8>(acc[mt], init, m0 + 16 * mt, n0);
    if (live(m0, n0)) {
      const int2 kr = krange(m0, n0);
      tile_mma<MT, NT8>(acc, fa, fb, m0, n0, kr.x, kr.y);
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) tile_epi<NT8>(acc[mt], epi, m0 + 16 * mt, n0);
  }
}
template <int M, int N, int NT8, class FA, class FB, class FL, class FR, class FI, class FE>
__device__ __forceinline__ void cta_gemm(const FA& fa, const FB& fb, const FL& live, const FR& krange, const FI& init,
                                         const FE& epi) {
  cta_gemm<M, N, NT8, 1>(fa, fb, live, krange, init, epi);
}

// ---------------------------------------------------------------- prep ----
template <int K, int V>
struct PrepSmem {
  static constexpr int LK = K + 4, LV = V + 4, LX = (K > V ? K : V) + 4;
  static constexpr int B0 = 0, B1 = B0 + C * LX, B2 = B1 + C * LX, B3 = B2 + C * LX, B4 = B3 + C * LX,
                       X1 = B4 + C * LX, X2 = X1 + C * LC, X3 = X2 + C * LC, F = X3 + C * LC, G = F + 4 * K,
                       D = G + 4 * K, EG = D + 10 * K, BS = EG + K, FLOATS = BS + C;
  // + an mbarrier and the TMEM slot after the floats, and up to 1 KB to align the base
  // (the 64 x (K + 4) buffers then start on 1 KB boundaries, as swizzled operands need)
  static constexpr int BYTES = FLOATS * 4 + 16 + 1024;
  static_assert(8 * K <= C * LC, "block references fit in the T tile");
  static_assert((C * LX * 4) % 1024 == 0 && (FLOATS * 4) % 8 == 0, "aligned buffers");
};
__device__ __forceinline__ int pair_index(int bi, int bj) { return bi * (bi + 1) / 2 + bj; }
// K = 128: the slot's Q region holds Q as two bf16 tiles (high part, then the low part
// at kQLow bytes), K-major with the 128-byte swizzle (64-column blocks of 128 rows)
constexpr uint32_t kQLow = 32768;

// q, k, g rows of a chunk -> gc (log2 units, in place of g), the block references
// (refs: s_b [4][N], e_b [4][N]) and the tables Lk = k e^{gc - s_b}, Lq = scale q e^{gc - s_b}
// (in place of k and q) and R = k e^{e_b - gc}.  Columns [0, N) of stride LD.
template <int N, int LD>
__device__ __forceinline__ void make_tables(float* kL, float* qL, float* gc, float* R, float* refs, float scale) {
  cumsum_log2<N, LD>(gc);
  __syncthreads();
  for (int idx = threadIdx.x; idx < 4 * N; idx += NT) {
    const int b = idx / N, d = idx - b * N;
    refs[4 * N + idx] = gc[(16 * b + 15) * LD + d];
    refs[idx] = b == 0 ? 0.f : gc[(16 * b - 1) * LD + d];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < C * N; idx += NT) {
    const int i = idx / N, d = idx - i * N, b = i >> 4;
    const float x = gc[i * LD + d], s = refs[b * N + d], e = refs[(4 + b) * N + d];
    const float kk = kL[i * LD + d];
    const float f = ex2(x - s);
    kL[i * LD + d] = kk * f;
    if (qL) qL[i * LD + d] = scale * qL[i * LD + d] * f;
    R[i * LD + d] = kk * ex2(e - x);
  }
}

// T = (I + M)^{-1}, M = strict_tril(Diag(beta) KKd), into Tm (C x C, stride LC): the
// 16 x 16 diagonal blocks by forward substitution, then block rows a > b level by level:
// T_ab = -T_aa sum_{c=b}^{a-1} M_ac T_cb.  tmp: 3 x 256 floats.
__device__ __forceinline__ void tri_inverse(const float* KKd, const float* bs, float* Tm, float* tmp) {
  const int tid = threadIdx.x;
  if (tid < 64) {
    const int bb = tid >> 4, jc = tid & 15, o = 16 * bb;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float s = (i == jc) ? 1.f : 0.f;
      const float bi = bs[o + i];
#pragma unroll
      for (int mm = 0; mm < i; ++mm) s = fmaf(-bi * KKd[(o + i) * LC + o + mm], acc[mm], s);
      acc[i] = s;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tm[(o + i) * LC + o + jc] = acc[i];
  }
  for (int idx = tid; idx < C * C; idx += NT) {
    const int r = idx >> 6, c = idx & 63;
    if ((c >> 4) > (r >> 4)) Tm[r * LC + c] = 0.f;
  }
  __syncthreads();
  for (int L = 1; L < 4; ++L) {
    const int nb = 4 - L;
    for (int idx = tid; idx < nb * 256; idx += NT) {
      const int b = idx >> 8, r = (idx >> 4) & 15, c = idx & 15, a = b + L;
      const float ba = bs[16 * a + r];
      float s = 0.f;
      for (int mm = 16 * b; mm < 16 * a; ++mm) s = fmaf(ba * KKd[(16 * a + r) * LC + mm], Tm[mm * LC + 16 * b + c], s);
      tmp[idx] = s;
    }
    __syncthreads();
    for (int idx = tid; idx < nb * 256; idx += NT) {
      const int b = idx >> 8, r = (idx >> 4) & 15, c = idx & 15, a = b + L;
      float s = 0.f;
      for (int mm = 0; mm <= r; ++mm) s = fmaf(Tm[(16 * a + r) * LC + 16 * a + mm], tmp[(b << 8) + (mm << 4) + c], s);
      Tm[(16 * a + r) * LC + 16 * b + c] = -s;
    }
    __syncthreads();
  }
}

// In place: the fp32 64 x 128 tile `buf` (row stride LD) -> its bf16 high and low parts as
// MN-major tcgen05 operands (K = the 64 rows, M or N = the 128 columns; 128-byte
// swizzle, 64-column atoms 8 KB apart; the high part at byte 0, the low part at 16 KB).
// val(i, c, x) gives the value of element (i, c) from its stored x.  Ends with a barrier
// before the writes only: the caller orders the writes with later readers.
template <int LD, class FV>
__device__ __forceinline__ void split_mn(float* buf, const FV& val) {
  float v[4][8];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = threadIdx.x + NT * u, i = c >> 4, n = (c & 15) << 3;
    const float4 a = *reinterpret_cast<const float4*>(buf + i * LD + n);
    const float4 b = *reinterpret_cast<const float4*>(buf + i * LD + n + 4);
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) v[u][e] = val(i, n + e, x[e]);
  }
  __syncthreads();
  uint8_t* base = reinterpret_cast<uint8_t*>(buf);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = threadIdx.x + NT * u, i = c >> 4, n = (c & 15) << 3;
    const uint32_t off = (n >> 6) * 8192u + (i >> 3) * 1024u + (i & 7) * 128u + ((((n & 63) >> 3) ^ (i & 7)) << 4);
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 hb = __floats2bfloat162_rn(v[u][2 * e], v[u][2 * e + 1]);
      const __nv_bfloat162 lb = __floats2bfloat162_rn(v[u][2 * e] - __low2float(hb), v[u][2 * e + 1] - __high2float(hb));
      h[e] = *reinterpret_cast<const uint32_t*>(&hb);
      l[e] = *reinterpret_cast<const uint32_t*>(&lb);
    }
    *reinterpret_cast<uint4*>(base + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(base + 16384 + off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}
// D[tmem] (=) A B for two split operands made by split_mn (A: M = 128 from its columns,
// B: N = 128 from its columns, K = 64 rows): Ah Bh + Ah Bl + Al Bh, issued by one thread.
__device__ __forceinline__ void issue_split_mn(uint32_t d_tmem, uint32_t a, uint32_t b) {
  constexpr uint32_t idesc = idesc_f16kind(128, 128) | IDESC_A_MN_MAJOR | IDESC_B_MN_MAJOR;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const uint64_t ah = sdesc(a + ks * 2048, 8192, 1024, 2), al = sdesc(a + 16384 + ks * 2048, 8192, 1024, 2);
    const uint64_t bh = sdesc(b + ks * 2048, 8192, 1024, 2), bl = sdesc(b + 16384 + ks * 2048, 8192, 1024, 2);
    umma_f16(d_tmem, ah, bh, idesc, ks > 0 ? 1u : 0u);
    umma_f16(d_tmem, ah, bl, idesc, 1u);
    umma_f16(d_tmem, al, bh, idesc, 1u);
  }
}

// prep_kernel's products with K = V = 128 (after W): Q = Diag(e^{gl}) - kr^T W,
// R = kr^T U and B = qd^T do - W^T E on tcgen05 (fp32 accumulators in 512 TMEM columns),
// from operands split in place; U and E by warp products in between.
template <typename IO>
__device__ __forceinline__ void prep_qrb_tc(const Params& p, float* sm, float* slot, long tok0, int rows, int hv,
                                            const float* X1, const float* X2, const float* X3, float* B0, float* B1,
                                            float* B2, float* B3, float* B4, const float* F, const float* G,
                                            const float* EG, const float* bs, uint64_t* mbar, uint32_t* tslot) {
  constexpr int K = 128, V = 128, LK = K + 4, LV = V + 4;
  using S = Slot<K, V>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const auto zero = [](int, int) { return 0.f; };
  const auto all = [](int, int) { return true; };
  const auto fa_A = [&](int i, int j, int) { return X3[i * LC + j] * bs[j]; };
  const auto kr_tril = [](int m0, int) { return make_int2(0, m0 + 32); };
  // W (fp32) to the slot, then W and kr = R e^{gl - e_b} split; Q's products
  copy_out<K, LK>(slot + S::W, B2);
  split_mn<LK>(B2, [](int, int, float x) { return x; });
  split_mn<LK>(B3, [&](int i, int d, float x) { return x * G[(i >> 4) * K + d]; });
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    issue_split_mn(tmem, smem_u32(B3), smem_u32(B2));
  }
  // U = A v (B4), to the slot, split; R's products
  load_rows<IO, V>(B0, static_cast<const IO*>(p.v), tok0, rows, static_cast<size_t>(p.HV) * V, static_cast<size_t>(hv) * V);
  __syncthreads();
  cta_gemm<C, V, 4, 2>(fa_A, [&](int j, int vv, int) { return B0[j * LV + vv]; }, all, kr_tril, zero,
                       [&](int r, int c, float x0, float x1) {
                         B4[r * LV + c] = x0;
                         B4[r * LV + c + 1] = x1;
                       });
  __syncthreads();
  copy_out<V, LV>(slot + S::U, B4);
  split_mn<LV>(B4, [](int, int, float x) { return x; });
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    issue_split_mn(tmem + 128, smem_u32(B3), smem_u32(B4));
    umma_commit(mbar);  // phase 0: Q and R
  }
  // E = Aqk^T do (B4 once R's products have read U), to the slot; do, E and qd split
  load_rows<IO, V>(B0, static_cast<const IO*>(p.d_out), tok0, rows, static_cast<size_t>(p.HV) * V,
                   static_cast<size_t>(hv) * V);
  if (!mbar_wait(mbar, 0, p.wait_ns)) {
    atomicOr(p.status, kStatusTimeout);
    mbar_wait(mbar, 0, kDrainNs);  // U is rewritten only once the products that read it are done
  }
  tc_fence_after();
  __syncthreads();
  cta_gemm<C, V, 4, 2>([&](int j, int i, int) { return X2[i * LC + j]; }, [&](int i, int vv, int) { return B0[i * LV + vv]; },
                       all, [](int m0, int) { return make_int2(m0, C); }, zero, [&](int r, int c, float x0, float x1) {
                         B4[r * LV + c] = x0;
                         B4[r * LV + c + 1] = x1;
                       });
  __syncthreads();
  copy_out<V, LV>(slot + S::E, B4);
  split_mn<LV>(B4, [](int, int, float x) { return x; });
  split_mn<LV>(B0, [](int, int, float x) { return x; });
  split_mn<LK>(B1, [&](int i, int d, float x) { return x * F[(i >> 4) * K + d]; });
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    issue_split_mn(tmem + 256, smem_u32(B1), smem_u32(B0));  // qd^T do
    issue_split_mn(tmem + 384, smem_u32(B2), smem_u32(B4));  // W^T E
    umma_commit(mbar);  // phase 1
  }
  copy_out<C, LC>(slot + S::T, X3);
  copy_out<C, LC>(slot + S::KK, X1);
  if (!mbar_wait(mbar, 1, p.wait_ns)) {
    atomicOr(p.status, kStatusTimeout);
    mbar_wait(mbar, 1, kDrainNs);  // the accumulators are read and released only after the products
  }
  tc_fence_after();
  // readout: warp w holds key rows 32 (w % 4) + lane, columns 64 (w / 4) + [0, 64).  Q, R
  // and B are staged in shared memory (free now: the operands' products are done, T and
  // kd ki^T are out) in their slot layouts, then written by three bulk copies.
  __syncthreads();  // every thread's copies of T and kd ki^T have read their tiles
  const int d = 32 * (warp & 3) + lane, h = warp >> 2;
  const uint32_t trow = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 64 * h;
  uint8_t* stq = reinterpret_cast<uint8_t*>(sm);  // [0, 64 KB): Q; [64, 128 KB): R; [128, 192 KB): B
  float* str = sm + 16384;
  float* stb = sm + 32768;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float x[32];
    tmem_ld32(trow + 32 * half, x);
    tmem_ld_wait();
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {  // Q: bf16 high / low parts, K-major 128-B swizzled
      const int e0 = 64 * h + 32 * half + 8 * c8;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = e0 + 2 * e;
        const float y0 = (d == c ? EG[d] : 0.f) - x[8 * c8 + 2 * e], y1 = (d == c + 1 ? EG[d] : 0.f) - x[8 * c8 + 2 * e + 1];
        const __nv_bfloat162 hb = __floats2bfloat162_rn(y0, y1);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(y0 - __low2float(hb), y1 - __high2float(hb));
        hi[e] = *reinterpret_cast<const uint32_t*>(&hb);
        lo[e] = *reinterpret_cast<const uint32_t*>(&lb);
      }
      const uint32_t o = sw128_offset(d, e0, K);
      *reinterpret_cast<uint4*>(stq + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(stq + kQLow + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float r[32], b1[32], b2[32];
    tmem_ld32(trow + 128 + 32 * half, r);
    tmem_ld32(trow + 256 + 32 * half, b1);
    tmem_ld32(trow + 384 + 32 * half, b2);
    tmem_ld_wait();
    float* rp = str + kv_off<K>(d, 64 * h + 32 * half);
    float* bp = stb + kv_off<K>(d, 64 * h + 32 * half);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      *reinterpret_cast<float4*>(rp + 4 * j) = make_float4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      *reinterpret_cast<float4*>(bp + 4 * j) = make_float4(b1[4 * j] - b2[4 * j], b1[4 * j + 1] - b2[4 * j + 1],
                                                           b1[4 * j + 2] - b2[4 * j + 2], b1[4 * j + 3] - b2[4 * j + 3]);
    }
  }
  fence_proxy_async_smem();  // the staged tiles (generic stores) before the bulk copies read them
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    bulk_store(slot + S::Q, stq, 65536);
    bulk_store(slot + S::RH, str, 65536);
    bulk_store(slot + S::BD, stb, 65536);
    bulk_commit();
    bulk_wait_read();  // shared memory is read before the CTA releases it
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <typename IO, int K, int V>
__global__ void __launch_bounds__(NT, 1) prep_kernel(Params p) {
  using S = Slot<K, V>;
  using L = PrepSmem<K, V>;
  constexpr int LK = L::LK, LV = L::LV;
  constexpr bool TC = K == 128 && V == 128;  // Q, R and B on tcgen05
  extern __shared__ __align__(16) uint8_t praw[];
  float* sm = reinterpret_cast<float*>(praw + ((1024u - (smem_u32(praw) & 1023u)) & 1023u));
  float *B0 = sm + L::B0, *B1 = sm + L::B1, *B2 = sm + L::B2, *B3 = sm + L::B3, *B4 = sm + L::B4;
  float *X1 = sm + L::X1, *X2 = sm + L::X2, *X3 = sm + L::X3;
  float *F = sm + L::F, *G = sm + L::G, *D = sm + L::D, *EG = sm + L::EG, *bs = sm + L::BS;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + L::FLOATS);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::FLOATS) + 2;
  int seq, m, rows;
  long tok0;
  const int f = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
  if (!find_chunk(p, f, seq, m, tok0, rows)) return;
  if constexpr (TC) {
    if (tid == 0) {
      mbar_init(mbar, 1);
      fence_mbar_init();
    }
    if (tid < 32) tmem_alloc(tslot, 512);
    tc_fence_before();
  }
  const int hk = hv / (p.HV / p.H);
  float* slot = p.ws + (static_cast<size_t>(f) * p.HV + hv) * p.slot_floats;
  const auto zero = [](int, int) { return 0.f; };
  const auto all = [](int, int) { return true; };

  // 1. rows of k, q, g; the tables (Lk in B0, Lq in B1, R in B3; gc in B2)
  load_rows<IO, K>(B0, static_cast<const IO*>(p.k), tok0, rows, static_cast<size_t>(p.H) * K, static_cast<size_t>(hk) * K);
  load_rows<IO, K>(B1, static_cast<const IO*>(p.q), tok0, rows, static_cast<size_t>(p.H) * K, static_cast<size_t>(hk) * K);
  load_rows<float, K>(B2, p.g, tok0, rows, static_cast<size_t>(p.HV) * K, static_cast<size_t>(hv) * K);
  if (tid < C) bs[tid] = tid < rows ? p.beta[(tok0 + tid) * p.HV + hv] : 0.f;
  __syncthreads();
  float* refs = X3;  // s_b, e_b until T is formed
  make_tables<K, LK>(B0, B1, B2, B3, refs, p.scale);
  for (int idx = tid; idx < 4 * K; idx += NT) {
    const int b = idx / K, d = idx - b * K;
    F[idx] = ex2(refs[idx]);                               // e^{s_b}
    G[idx] = ex2(refs[7 * K + d] - refs[(4 + b) * K + d]);  // e^{gl - e_b}
    if (b == 0) EG[d] = ex2(refs[7 * K + d]);               // e^{gl}
  }
  for (int idx = tid; idx < 4 * K; idx += NT)
    if (!(refs[4 * K + idx] - refs[idx] >= kMinBlockLog2)) atomicOr(p.status, kStatusRange);
  for (int idx = tid; idx < 10 * K; idx += NT) {
    const int pr = idx / K, d = idx - pr * K;
    const int bi = pr >= 6 ? 3 : pr >= 3 ? 2 : pr >= 1 ? 1 : 0, bj = pr - bi * (bi + 1) / 2;
    D[idx] = ex2(refs[bi * K + d] - refs[(4 + bj) * K + d]);  // e^{s_bi - e_bj}, bj <= bi
  }
  __syncthreads();

  // 2. KKd = strict_tril(kd ki^T) (X1) and Aqk = tril(qd ki^T) (X2), block by block:
  //    (i, j) in blocks (bi, bj): sum_d Lk_i e^{s_bi - e_bj} R_j
  {
    const auto rb = [&](int kk, int nn, int) { return B3[nn * LK + kk]; };
    const auto lower = [](int m0, int n0) { return n0 <= m0 + 16; };
    const auto kr = [](int, int) { return make_int2(0, K); };
    cta_gemm<C, C, 2, 2>([&](int mm, int kk, int n0) { return B0[mm * LK + kk] * D[pair_index(mm >> 4, n0 >> 4) * K + kk]; },
                      rb, lower, kr, zero, [&](int r, int c, float x0, float x1) {
                        X1[r * LC + c] = c < r ? x0 : 0.f;
                        X1[r * LC + c + 1] = c + 1 < r ? x1 : 0.f;
                      });
    cta_gemm<C, C, 2, 2>([&](int mm, int kk, int n0) { return B1[mm * LK + kk] * D[pair_index(mm >> 4, n0 >> 4) * K + kk]; },
                      rb, lower, kr, zero, [&](int r, int c, float x0, float x1) {
                        X2[r * LC + c] = c <= r ? x0 : 0.f;
                        X2[r * LC + c + 1] = c + 1 <= r ? x1 : 0.f;
                      });
  }
  __syncthreads();
  // 3. T (X3), with B2's first 768 floats as scratch (gc is no longer needed)
  tri_inverse(X1, bs, X3, B2);
  // 4. W = A kd (B2): A = T Diag(beta), kd = Lk e^{s_b}
  const auto fa_A = [&](int i, int j, int) { return X3[i * LC + j] * bs[j]; };
  const auto kr_tril = [](int m0, int) { return make_int2(0, m0 + 32); };
  cta_gemm<C, K, 4, 2>(fa_A, [&](int j, int d, int) { return B0[j * LK + d] * F[(j >> 4) * K + d]; }, all, kr_tril, zero,
                    [&](int r, int c, float x0, float x1) {
                      B2[r * LK + c] = x0;
                      B2[r * LK + c + 1] = x1;
                    });
  __syncthreads();
  if constexpr (TC) {
    prep_qrb_tc<IO>(p, sm, slot, tok0, rows, hv, X1, X2, X3, B0, B1, B2, B3, B4, F, G, EG, bs, mbar, tslot);
    return;
  }
  // 5. Q = Diag(e^{gl}) - kr^T W (kr = R e^{gl - e_b}); W to the slot
  const auto fa_krT = [&](int d, int i, int) { return B3[i * LK + d] * G[(i >> 4) * K + d]; };
  const auto kr_all = [](int, int) { return make_int2(0, C); };
  cta_gemm<K, K, 4, 2>(fa_krT, [&](int i, int e, int) { return B2[i * LK + e]; }, all, kr_all, zero,
                    [&](int r, int c, float x0, float x1) {
                      const float y0 = (r == c ? EG[r] : 0.f) - x0, y1 = (r == c + 1 ? EG[r] : 0.f) - x1;
                      if (K == 128) {  // bf16 high / low parts, K-major 128-B swizzled (the tcgen05 chain's A)
                        uint8_t* qb = reinterpret_cast<uint8_t*>(slot + S::Q);
                        const uint32_t o = sw128_offset(r, c, K);
                        const __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
                        const __nv_bfloat162 l =
                            __floats2bfloat162_rn(y0 - __low2float(h), y1 - __high2float(h));
                        *reinterpret_cast<__nv_bfloat162*>(qb + o) = h;
                        *reinterpret_cast<__nv_bfloat162*>(qb + kQLow + o) = l;
                      } else {
                        *reinterpret_cast<float2*>(slot + S::Q + static_cast<size_t>(r) * K + c) = make_float2(y0, y1);
                      }
                    });
  copy_out<K, LK>(slot + S::W, B2);
  __syncthreads();
  // 6. U = A v (B4), R = kr^T U to the slot
  load_rows<IO, V>(B0, static_cast<const IO*>(p.v), tok0, rows, static_cast<size_t>(p.HV) * V, static_cast<size_t>(hv) * V);
  __syncthreads();
  cta_gemm<C, V, 4, 2>(fa_A, [&](int j, int vv, int) { return B0[j * LV + vv]; }, all, kr_tril, zero,
                    [&](int r, int c, float x0, float x1) {
                      B4[r * LV + c] = x0;
                      B4[r * LV + c + 1] = x1;
                    });
  __syncthreads();
  cta_gemm<K, V, 4, 2>(fa_krT, [&](int i, int vv, int) { return B4[i * LV + vv]; }, all, kr_all, zero,
                    [&](int r, int c, float x0, float x1) {
                      *reinterpret_cast<float2*>(slot + S::RH + kv_off<K>(r, c)) = make_float2(x0, x1);
                    });
  copy_out<V, LV>(slot + S::U, B4);
  __syncthreads();
  // 7. E = Aqk^T do (B4), B = qd^T do - W^T E to the slot
  load_rows<IO, V>(B0, static_cast<const IO*>(p.d_out), tok0, rows, static_cast<size_t>(p.HV) * V,
                   static_cast<size_t>(hv) * V);
  __syncthreads();
  cta_gemm<C, V, 4, 2>([&](int j, int i, int) { return X2[i * LC + j]; }, [&](int i, int vv, int) { return B0[i * LV + vv]; },
                    all, [](int m0, int) { return make_int2(m0, C); }, zero, [&](int r, int c, float x0, float x1) {
                      B4[r * LV + c] = x0;
                      B4[r * LV + c + 1] = x1;
                    });
  __syncthreads();
  cta_gemm<K, V, 4, 2>(
      [&](int d, int kk, int) { return kk < C ? B1[kk * LK + d] * F[(kk >> 4) * K + d] : -B2[(kk - C) * LK + d]; },
      [&](int kk, int vv, int) { return kk < C ? B0[kk * LV + vv] : B4[(kk - C) * LV + vv]; }, all,
      [](int, int) { return make_int2(0, 2 * C); }, zero, [&](int r, int c, float x0, float x1) {
        *reinterpret_cast<float2*>(slot + S::BD + kv_off<K>(r, c)) = make_float2(x0, x1);
      });
  copy_out<V, LV>(slot + S::E, B4);
  copy_out<C, LC>(slot + S::T, X3);
  copy_out<C, LC>(slot + S::KK, X1);
}

// --------------------------------------------------------------- chains ----
// One CTA per 64 value columns and direction: X (K x 64, two buffers) in shared memory,
// Q of the next chunk prefetched by cp.async while the current one is applied, the
// addend (R or B) read straight into the accumulators' registers.
constexpr int VS = 64;  // value columns per chain CTA
template <int K>
struct ChainSmem {
  static constexpr int LK = K + 4, LS = VS + 4;
  static constexpr int Q0 = 0, Q1 = K * LK, X0 = 2 * K * LK, X1 = X0 + K * LS, FLOATS = X1 + K * LS;
};
template <int K, int V>
__global__ void __launch_bounds__(NT, 1) chain_kernel(Params p) {
  using S = Slot<K, V>;
  using L = ChainSmem<K>;
  constexpr int LK = L::LK, LS = L::LS;
  constexpr int VC = V < VS ? V : VS;       // value columns of this CTA
  constexpr int RB = K / 16;                // 16-row blocks of the K x VC product
  constexpr int WPR = NW / RB;              // warps per row block
  constexpr int NT8 = VC / (8 * WPR);       // one 16 x (8 NT8) tile per warp
  static_assert(NW % RB == 0 && VC % (8 * WPR) == 0, "tiles");
  extern __shared__ __align__(16) float sm[];
  auto Qb = [&](int b) { return sm + (b ? L::Q1 : L::Q0); };
  auto Xb = [&](int b) { return sm + (b ? L::X1 : L::X0); };
  const int v0 = blockIdx.x * VC, hv = blockIdx.y, seq = blockIdx.z >> 1, dir = blockIdx.z & 1, tid = threadIdx.x;
  int f0, nch;
  if (!seq_chunks(p, seq, f0, nch)) return;
  const float* x0 = dir == 0 ? p.s0 : p.d_fin;
  const size_t state0 = (static_cast<size_t>(seq) * p.HV + hv) * K * V + v0;
  for (int idx = tid; idx < K * VC; idx += NT) {
    const int r = idx / VC, c = idx - r * VC;
    Xb(0)[r * LS + c] = x0 ? x0[state0 + static_cast<size_t>(r) * V + c] : 0.f;
  }
  const size_t add = dir == 0 ? S::RH : S::BD;
  auto slot = [&](int step) {
    return p.ws + (static_cast<size_t>(f0 + (dir == 0 ? step : nch - 1 - step)) * p.HV + hv) * p.slot_floats;
  };
  auto issue = [&](int step, int buf) {
    const float* s = slot(step);
    for (int idx = tid; idx < K * (K / 4); idx += NT) {
      const int r = idx / (K / 4), c4 = (idx - r * (K / 4)) * 4;
      cp_async16(Qb(buf) + r * LK + c4, s + S::Q + static_cast<size_t>(r) * K + c4);
    }
    cp_async_commit();
  };
  if (nch > 0) issue(0, 0);
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int m0 = 16 * (warp / WPR), n0 = (warp % WPR) * 8 * NT8;
  int cur = 0;
  for (int step = 0; step < nch; ++step) {
    float* s = slot(step);
    if (step + 1 < nch) {
      issue(step + 1, (step + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // Q of this chunk and X visible to every thread
    float2 ad[NT8][2];  // this tile's addend
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        ad[nt][h] = *reinterpret_cast<const float2*>(s + add + kv_off<K>(m0 + g + 8 * h, v0 + n0 + 8 * nt + 2 * t));
    const float* Q = Qb(step & 1);
    const float* X = Xb(cur);
    float acc[NT8][4];
    tile_init<NT8>(acc, [](int, int) { return 0.f; }, m0, n0);
    if (dir == 0)
      tile_mma<NT8>(acc, [&](int d, int e, int) { return Q[d * LK + e]; }, [&](int e, int c, int) { return X[e * LS + c]; },
                    m0, n0, 0, K);
    else
      tile_mma<NT8>(acc, [&](int d, int e, int) { return Q[e * LK + d]; }, [&](int e, int c, int) { return X[e * LS + c]; },
                    m0, n0, 0, K);
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
      acc[nt][0] += ad[nt][0].x;
      acc[nt][1] += ad[nt][0].y;
      acc[nt][2] += ad[nt][1].x;
      acc[nt][3] += ad[nt][1].y;
    }
    __syncthreads();  // every thread has its addend: the slot's addend place may be overwritten
    // the state entering the chunk (forward) / the gradient leaving it (reverse)
    for (int idx = tid; idx < K * (VC / 4); idx += NT) {
      const int r = idx / (VC / 4), c4 = (idx - r * (VC / 4)) * 4;
      *reinterpret_cast<float4*>(s + add + kv_off<K>(r, v0 + c4)) =
          *reinterpret_cast<const float4*>(X + r * LS + c4);
    }
    float* Xn = Xb(cur ^ 1);
    tile_epi<NT8>(acc, [&](int r, int c, float a, float b) { *reinterpret_cast<float2*>(Xn + r * LS + c) = make_float2(a, b); },
                  m0, n0);
    cur ^= 1;
  }
  if (dir == 1 && p.ds0) {
    __syncthreads();
    const float* X = Xb(cur);
    for (int idx = tid; idx < K * VC; idx += NT) {
      const int r = idx / VC, c = idx - r * VC;
      p.ds0[state0 + static_cast<size_t>(r) * V + c] = X[r * LS + c];
    }
  }
}

// ------------------------------------------------------ chains (tcgen05) ----
// K = 128.  The CTA's 64 value columns of X are the fp32 accumulator of a tcgen05 product
// in TMEM (lane = key row, 64 columns).  Per chunk: D = addend (tcgen05.st) +
// Q X (forward) or Q^T X (reverse) as the three bf16 products Qh Xh + Qh Xl + Ql Xh of
// the high/low splits (M = 128, N = 64, K = 128).  Q's splits arrive by bulk copy two
// chunks ahead; the same K-major tiles are Q^T as MN-major A operands.  X's splits are
// written back to shared memory (MN-major B, 128-byte swizzle) after each product.
namespace tcc {
constexpr uint32_t QBUF = 65536;                       // Q high + low
constexpr uint32_t ABUF = 32768;                       // the addend slice, 128 x 64 fp32
constexpr uint32_t BUF = QBUF + ABUF;
constexpr uint32_t XH = 2 * BUF, XL = XH + 16384, BAR = XL + 16384, SMEM = BAR + 64 + 1024;
}  // namespace tcc
template <int V>
__global__ void __launch_bounds__(NT, 1) chain_tc_kernel(Params p) {
  constexpr int K = 128, VC = 64;
  using S = Slot<K, V>;
  extern __shared__ __align__(16) uint8_t smraw[];
  uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + tcc::BAR);  // [0], [1]: buffer full; [2]: products done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + tcc::BAR + 32);
  volatile uint32_t* failed = reinterpret_cast<volatile uint32_t*>(sm + tcc::BAR + 40);
  const int v0 = blockIdx.x * VC, hv = blockIdx.y, seq = blockIdx.z >> 1, dir = blockIdx.z & 1, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int f0, nch;
  if (!seq_chunks(p, seq, f0, nch)) return;
  const int row = 32 * (warp & 3) + lane, c0 = 32 * (warp >> 2);  // this thread's key row and 32 columns
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    *failed = 0u;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot, tm_row = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + c0;
  const uint32_t sb = smem_u32(sm);
  const size_t add = (dir == 0 ? S::RH : S::BD) + kv_off<K>(0, v0);  // this CTA's 128 x 64 slice
  auto slot = [&](int step) {
    return p.ws + (static_cast<size_t>(f0 + (dir == 0 ? step : nch - 1 - step)) * p.HV + hv) * p.slot_floats;
  };
  auto issue = [&](int step) {  // thread 0: Q and the addend slice of this step's chunk into buffer step & 1
    const float* s = slot(step);
    const uint8_t* qs = reinterpret_cast<const uint8_t*>(s + S::Q);
    const uint8_t* as = reinterpret_cast<const uint8_t*>(s + add);
    uint8_t* dst = sm + (step & 1) * tcc::BUF;
    mbar_arrive_expect_tx(&bars[step & 1], tcc::BUF);
#pragma unroll
    for (int q = 0; q < 4; ++q) bulk_load(dst + q * 16384, qs + q * 16384, 16384, &bars[step & 1]);
#pragma unroll
    for (int q = 0; q < 2; ++q) bulk_load(dst + tcc::QBUF + q * 16384, as + q * 16384, 16384, &bars[step & 1]);
  };
  auto put_x = [&](const float (&x)[32]) {  // X's splits for the next product (key row `row`)
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      uint32_t h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 hb = __floats2bfloat162_rn(x[8 * j8 + 2 * e], x[8 * j8 + 2 * e + 1]);
        const __nv_bfloat162 lb =
            __floats2bfloat162_rn(x[8 * j8 + 2 * e] - __low2float(hb), x[8 * j8 + 2 * e + 1] - __high2float(hb));
        h[e] = *reinterpret_cast<const uint32_t*>(&hb);
        l[e] = *reinterpret_cast<const uint32_t*>(&lb);
      }
      const uint32_t off = (row >> 3) * 1024u + (row & 7) * 128u + ((((c0 >> 3) + j8) ^ (row & 7)) << 4);
      *reinterpret_cast<uint4*>(sm + tcc::XH + off) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(sm + tcc::XL + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
  };
  float x[32];
  {
    const float* x0 = dir == 0 ? p.s0 : p.d_fin;
    const float* xp = x0 ? x0 + (static_cast<size_t>(seq) * p.HV + hv) * K * V + static_cast<size_t>(row) * V + v0 + c0 : nullptr;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v4 = xp ? *reinterpret_cast<const float4*>(xp + 4 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
      x[4 * j] = v4.x;
      x[4 * j + 1] = v4.y;
      x[4 * j + 2] = v4.z;
      x[4 * j + 3] = v4.w;
    }
  }
  put_x(x);
  int issued = nch < 2 ? nch : 2;  // steps [0, issued) have had their loads issued (thread 0's count)
  bool pending = false;            // products committed and not yet seen complete (thread 0)
  if (tid == 0)
    for (int s2 = 0; s2 < issued; ++s2) issue(s2);
  // descriptors of the k = 0 step (16-byte units added per step): A = Q's splits (K-major,
  // or MN-major for Q^T), B = X's splits (MN-major)
  const uint32_t idesc = idesc_f16kind(128, 64) | IDESC_B_MN_MAJOR | (dir ? IDESC_A_MN_MAJOR : 0u);
  const uint64_t dq0 = dir == 0 ? sdesc_sw128(sb) : sdesc(sb, 16384, 1024, 2);
  const uint64_t dxh = sdesc(sb + tcc::XH, 16384, 1024, 2), dxl = sdesc(sb + tcc::XL, 16384, 1024, 2);
  int step = 0;
  for (; step < nch; ++step) {
    const int b = step & 1;
    const uint8_t* buf = sm + b * tcc::BUF;
    // this chunk's Q and addend have landed (every thread reads the addend)
    if (!mbar_wait(&bars[b], (step >> 1) & 1, p.wait_ns)) {
      atomicOr(p.status, kStatusTimeout);
      *failed = 1u;
    }
    // the addend into D; the state entering the chunk (forward) / the gradient leaving
    // it (reverse) into the addend's place in the slot (its bulk read has completed)
    float a[32];
    const float* as = reinterpret_cast<const float*>(buf + tcc::QBUF) + row * 64 + c0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v4 = *reinterpret_cast<const float4*>(as + 4 * j);
      a[4 * j] = v4.x;
      a[4 * j + 1] = v4.y;
      a[4 * j + 2] = v4.z;
      a[4 * j + 3] = v4.w;
    }
    tmem_st32(tm_row, a);
    float* ap = slot(step) + add + row * 64 + c0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(ap + 4 * j) = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    tmem_st_wait();
    fence_proxy_async_smem();  // X's splits (generic stores) before the products read them
    tc_fence_before();
    __syncthreads();
    if (*failed) break;
    if (tid == 0) {
      tc_fence_after();
      const uint64_t qh = dq0 + ((b * tcc::BUF) >> 4), ql = qh + (kQLow >> 4);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ao = dir == 0 ? ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4 : (ks * 2048) >> 4;
        const uint32_t bo = (ks * 2048) >> 4;
        umma_f16(tmem, qh + ao, dxh + bo, idesc, 1u);
        umma_f16(tmem, qh + ao, dxl + bo, idesc, 1u);
        umma_f16(tmem, ql + ao, dxh + bo, idesc, 1u);
      }
      umma_commit(&bars[2]);
      pending = true;
    }
    if (mbar_wait(&bars[2], step & 1, p.wait_ns)) {
      pending = false;
    } else {
      atomicOr(p.status, kStatusTimeout);
      *failed = 1u;
    }
    tc_fence_after();
    __syncthreads();  // every thread has seen the products complete (or the failure) and read its addend
    if (*failed) break;
    if (tid == 0 && step + 2 < nch) {
      issue(step + 2);
      issued = step + 3;
    }
    tmem_ld32(tm_row, x);
    tmem_ld_wait();
    put_x(x);
  }
  if (tid == 0 && step < nch) {  // after a failure: the loads issued for later steps, and the products,
                                 // complete (bounded waits) before the CTA releases its memory
    for (int s2 = step; s2 < issued; ++s2) mbar_wait(&bars[s2 & 1], (s2 >> 1) & 1, kDrainNs);
    if (pending) mbar_wait(&bars[2], step & 1, kDrainNs);
  }
  if (dir == 1 && p.ds0 && !*failed) {
    float* dp = p.ds0 + (static_cast<size_t>(seq) * p.HV + hv) * K * V + static_cast<size_t>(row) * V + v0 + c0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(dp + 4 * j) = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// -------------------------------------------------------- value gradients --
constexpr int SR = 16;  // rows of S and dS' per streamed slice
template <int K, int V>
struct GvSmem {
  static constexpr int LK = K + 4, LV = V + 4, LX = (K > V ? K : V) + 4;
  static constexpr int B0 = 0, B1 = B0 + C * LX, B2 = B1 + C * LX, B3 = B2 + C * LX, B4 = B3 + C * LX,
                       H0 = B4 + C * LX, H1 = H0 + SR * LV, D0 = H1 + SR * LV, D1 = D0 + SR * LV, GL = D1 + SR * LV,
                       BS = GL + K, FLOATS = BS + C;
};
template <typename IO, int K, int V>
__global__ void __launch_bounds__(NT, 1) grad_v_kernel(Params p) {
  using S = Slot<K, V>;
  using L = GvSmem<K, V>;
  constexpr int LK = L::LK, LV = L::LV;
  constexpr int NT8 = V / 32;  // v_new / dv_new: one 32 x (V / 4) tile per warp
  extern __shared__ __align__(16) float sm[];
  float *B0 = sm + L::B0, *B1 = sm + L::B1, *B2 = sm + L::B2, *B3 = sm + L::B3, *B4 = sm + L::B4;
  auto Hs = [&](int b) { return sm + (b ? L::H1 : L::H0); };
  auto Ds = [&](int b) { return sm + (b ? L::D1 : L::D0); };
  float *gl2 = sm + L::GL, *bs = sm + L::BS;
  int seq, m, rows;
  long tok0;
  const int f = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!find_chunk(p, f, seq, m, tok0, rows)) return;
  const int hk = hv / (p.HV / p.H);
  float* slot = p.ws + (static_cast<size_t>(f) * p.HV + hv) * p.slot_floats;
  const auto zero = [](int, int) { return 0.f; };
  const auto all = [](int, int) { return true; };

  // 1. W (B0), U (B2), E (B3) from the slot, do (B4); kr = k e^{gl - gc} (B1)
  copy_in<K, LK>(B0, slot + S::W);
  copy_in<V, LV>(B3, slot + S::E);
  load_rows<IO, V>(B4, static_cast<const IO*>(p.d_out), tok0, rows, static_cast<size_t>(p.HV) * V, static_cast<size_t>(hv) * V);
  load_rows<float, K>(B1, p.g, tok0, rows, static_cast<size_t>(p.HV) * K, static_cast<size_t>(hv) * K);
  load_rows<IO, K>(B2, static_cast<const IO*>(p.k), tok0, rows, static_cast<size_t>(p.H) * K, static_cast<size_t>(hk) * K);
  __syncthreads();
  cumsum_log2<K, LK>(B1);
  __syncthreads();
  if (tid < K) gl2[tid] = B1[(C - 1) * LK + tid];
  __syncthreads();
  for (int idx = tid; idx < C * K; idx += NT) {
    const int i = idx / K, d = idx - i * K;
    B1[i * LK + d] = B2[i * LK + d] * ex2(gl2[d] - B1[i * LK + d]);
  }
  __syncthreads();
  copy_in<V, LV>(B2, slot + S::U);
  // slices of S (entering) and dS' (leaving) in SR-row pieces
  const float* hsrc = slot + S::RH;
  const float* dsrc = slot + S::BD;
  auto issue = [&](int sl, int buf) {
    for (int idx = tid; idx < SR * (V / 4); idx += NT) {
      const int r = idx / (V / 4), c4 = (idx - r * (V / 4)) * 4;
      const size_t o = kv_off<K>(sl * SR + r, c4);
      cp_async16(Hs(buf) + r * LV + c4, hsrc + o);
      cp_async16(Ds(buf) + r * LV + c4, dsrc + o);
    }
    cp_async_commit();
  };
  constexpr int NSL = K / SR;
  const int vm0 = 32 * (warp >> 2), vn0 = (V / 4) * (warp & 3);
  float avn[2][NT8][4], adv[2][NT8][4];
  // 2. pass 1: v_new = U - W S, dv_new = E + kr dS', DH = do S^T, dgl = e^{gl} sum_v S dS'
  __syncthreads();
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    tile_init<NT8>(avn[mt], [&](int r, int c) { return B2[r * LV + c]; }, vm0 + 16 * mt, vn0);
    tile_init<NT8>(adv[mt], [&](int r, int c) { return B3[r * LV + c]; }, vm0 + 16 * mt, vn0);
  }
  issue(0, 0);
  for (int sl = 0; sl < NSL; ++sl) {
    const int buf = sl & 1;
    if (sl + 1 < NSL) {
      issue(sl + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* h = Hs(buf);
    const float* ds = Ds(buf);
    const int d0 = sl * SR;
    tile_mma<2, NT8>(avn, [&](int i, int kk, int) { return -B0[i * LK + d0 + kk]; },
                  [&](int kk, int vv, int) { return h[kk * LV + vv]; }, vm0, vn0, 0, SR);
    tile_mma<2, NT8>(adv, [&](int i, int kk, int) { return B1[i * LK + d0 + kk]; },
                  [&](int kk, int vv, int) { return ds[kk * LV + vv]; }, vm0, vn0, 0, SR);
    {  // DH[:, slice]: 8 tiles of 16 x 8
      float a1[1][4] = {{0.f, 0.f, 0.f, 0.f}};
      const int m0 = 16 * (warp >> 1), n0 = 8 * (warp & 1);
      tile_mma<1>(a1, [&](int i, int vv, int) { return B4[i * LV + vv]; }, [&](int vv, int dd, int) { return h[dd * LV + vv]; },
                  m0, n0, 0, V);
      tile_epi<1>(a1, [&](int r, int c, float x0, float x1) {
        *reinterpret_cast<float2*>(slot + S::DH + static_cast<size_t>(r) * K + d0 + c) = make_float2(x0, x1);
      }, m0, n0);
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {  // dgl for rows 2 warp, 2 warp + 1 of the slice
      const int r = 2 * warp + rr;
      float s = 0.f;
      for (int vv = lane; vv < V; vv += 32) s = fmaf(h[r * LV + vv], ds[r * LV + vv], s);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
      if (lane == 0) slot[S::DGL + d0 + r] = ex2(gl2[d0 + r]) * s;
    }
    __syncthreads();  // the slice buffers may be refilled
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    tile_epi<NT8>(avn[mt], [&](int r, int c, float x0, float x1) {
      *reinterpret_cast<float2*>(B2 + r * LV + c) = make_float2(x0, x1);
    }, vm0 + 16 * mt, vn0);
    tile_epi<NT8>(adv[mt], [&](int r, int c, float x0, float x1) {
      *reinterpret_cast<float2*>(B3 + r * LV + c) = make_float2(x0, x1);
    }, vm0 + 16 * mt, vn0);
  }
  // 3. pass 2: dW = -dv_new S^T, dkr = v_new dS'^T
  issue(0, 0);
  for (int sl = 0; sl < NSL; ++sl) {
    const int buf = sl & 1;
    if (sl + 1 < NSL) {
      issue(sl + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // (first slice: v_new and dv_new written too)
    const float* h = Hs(buf);
    const float* ds = Ds(buf);
    const int d0 = sl * SR;
    const int m0 = 16 * (warp >> 1), n0 = 8 * (warp & 1);
    float a1[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    tile_mma<1>(a1, [&](int i, int vv, int) { return -B3[i * LV + vv]; }, [&](int vv, int dd, int) { return h[dd * LV + vv]; },
                m0, n0, 0, V);
    tile_epi<1>(a1, [&](int r, int c, float x0, float x1) {
      *reinterpret_cast<float2*>(slot + S::DW + static_cast<size_t>(r) * K + d0 + c) = make_float2(x0, x1);
    }, m0, n0);
    float a2[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    tile_mma<1>(a2, [&](int i, int vv, int) { return B2[i * LV + vv]; }, [&](int vv, int dd, int) { return ds[dd * LV + vv]; },
                m0, n0, 0, V);
    tile_epi<1>(a2, [&](int r, int c, float x0, float x1) {
      *reinterpret_cast<float2*>(slot + S::DKR + static_cast<size_t>(r) * K + d0 + c) = make_float2(x0, x1);
    }, m0, n0);
    __syncthreads();
  }
  // 4. v (B0), T (B1); dAqk = tril(do v_new^T), dAv = tril(dv_new v^T), dv = A^T dv_new
  load_rows<IO, V>(B0, static_cast<const IO*>(p.v), tok0, rows, static_cast<size_t>(p.HV) * V, static_cast<size_t>(hv) * V);
  copy_in<C, LC>(B1, slot + S::T);
  if (tid < C) bs[tid] = tid < rows ? p.beta[(tok0 + tid) * p.HV + hv] : 0.f;
  __syncthreads();
  const auto lower = [](int m0, int n0) { return n0 <= m0 + 16; };
  const auto kv = [](int, int) { return make_int2(0, V); };
  cta_gemm<C, C, 2, 2>([&](int i, int vv, int) { return B4[i * LV + vv]; }, [&](int vv, int j, int) { return B2[j * LV + vv]; },
                    lower, kv, zero, [&](int r, int c, float x0, float x1) {
                      *reinterpret_cast<float2*>(slot + S::DAQK + r * C + c) =
                          make_float2(c <= r ? x0 : 0.f, c + 1 <= r ? x1 : 0.f);
                    });
  cta_gemm<C, C, 2, 2>([&](int i, int vv, int) { return B3[i * LV + vv]; }, [&](int vv, int j, int) { return B0[j * LV + vv]; },
                    lower, kv, zero, [&](int r, int c, float x0, float x1) {
                      *reinterpret_cast<float2*>(slot + S::DAV + r * C + c) =
                          make_float2(c <= r ? x0 : 0.f, c + 1 <= r ? x1 : 0.f);
                    });
  cta_gemm<C, V, 4, 2>([&](int j, int i, int) { return B1[i * LC + j] * bs[j]; }, [&](int i, int vv, int) { return B3[i * LV + vv]; },
                    all, [](int m0, int) { return make_int2(m0, C); }, zero, [&](int r, int c, float x0, float x1) {
                      if (r < rows)
                        *reinterpret_cast<float2*>(p.dv + (static_cast<size_t>(tok0 + r) * p.HV + hv) * V + c) =
                            make_float2(x0, x1);
                    });
}

// ------------------------------------------------- value gradients (tcgen05) --
// K = V = 128: every product of grad_v_kernel as a transposed M = 128 tcgen05 product of
// bf16 high/low operand splits (three products each), fp32 accumulators in TMEM:
//   -v_new^T = h^T W^T - U^T   dv_new^T = D^T kr^T + E^T   DH^T = h do^T
//   -dW^T = h dv_new^T         dkr^T = D v_new^T
//   [do; dv_new] [v_new; v]^T: rows 0-63 x columns 0-63 are dAqk, rows 64-127 x 64-127 dAv
//   dv^T = dv_new^T (T Diag(beta))
// h (the state entering the chunk) and D (the gradient leaving it) stay in shared memory
// as split K-major tiles, which are also their transposes' MN-major tiles.
namespace gvt {
constexpr uint32_t RH = 0, RD = 65536, RW = 131072, RKR = 163840, RDO = 196608, RB = 229376;  // byte offsets
constexpr uint32_t SMEM = RB + 16 + 4 * (128 + 64) + 1024;
}  // namespace gvt
template <class FAH, class FAL, class FBH, class FBL>
__device__ __forceinline__ void issue_split(uint32_t d, const FAH& ah, const FAL& al, const FBH& bh, const FBL& bl,
                                            uint32_t idesc, int nks, bool accumulate) {
  for (int ks = 0; ks < nks; ++ks) {
    umma_f16(d, ah(ks), bh(ks), idesc, (accumulate || ks > 0) ? 1u : 0u);
    umma_f16(d, ah(ks), bl(ks), idesc, 1u);
    umma_f16(d, al(ks), bh(ks), idesc, 1u);
  }
}
// 8 fp32 values -> their bf16 high and low parts, as two 16-byte chunks
__device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    const __nv_bfloat162 lb = __floats2bfloat162_rn(x[2 * e] - __low2float(hb), x[2 * e + 1] - __high2float(hb));
    h[e] = *reinterpret_cast<const uint32_t*>(&hb);
    l[e] = *reinterpret_cast<const uint32_t*>(&lb);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
// byte offset of the 8-element chunk (row r, columns c8 .. c8 + 7) in a 128-byte-swizzled
// tile of 128-byte rows (one 64-column block; a K-major tile's row, an MN-major tile's K-row)
__device__ __forceinline__ uint32_t sw_chunk(uint32_t r, uint32_t c8) {
  return (r >> 3) * 1024u + (r & 7) * 128u + ((((c8 & 63) >> 3) ^ (r & 7)) << 4);
}
template <typename IO>
__global__ void __launch_bounds__(NT, 1) grad_v_tc_kernel(Params p) {
  constexpr int K = 128, V = 128, LK = K + 4;
  using S = Slot<K, V>;
  extern __shared__ __align__(16) uint8_t graw[];
  uint8_t* sm = graw + ((1024u - (smem_u32(graw) & 1023u)) & 1023u);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + gvt::RB);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + gvt::RB + 8);
  float* gl2 = reinterpret_cast<float*>(sm + gvt::RB + 16);
  float* bs = gl2 + K;
  int seq, m, rows;
  long tok0;
  const int f = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (!find_chunk(p, f, seq, m, tok0, rows)) return;
  const int hk = hv / (p.HV / p.H);
  float* slot = p.ws + (static_cast<size_t>(f) * p.HV + hv) * p.slot_floats;
  if (tid == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot, sb = smem_u32(sm);
  const int row = 32 * (warp & 3) + lane, hcol = 32 * (warp >> 2);  // TMEM lane; 32 of a 64-column block
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + hcol;
  uint32_t phase = 0;
  auto wait_products = [&]() {
    if (!mbar_wait(mbar, phase & 1, p.wait_ns)) {
      atomicOr(p.status, kStatusTimeout);
      mbar_wait(mbar, phase & 1, kDrainNs);
    }
    ++phase;
    tc_fence_after();
  };
  const IO* dop = static_cast<const IO*>(p.d_out);
  const IO* vp = static_cast<const IO*>(p.v);
  const size_t vrow = static_cast<size_t>(p.HV) * V, vcol = static_cast<size_t>(hv) * V;

  // 1. kr = k e^{gl - gc} from g and k rows (fp32 scratch over the h, D regions), split
  //    K-major; beta
  {
    float* gs = reinterpret_cast<float*>(sm);
    float* ks_ = gs + C * LK;
    load_rows<float, K>(gs, p.g, tok0, rows, static_cast<size_t>(p.HV) * K, static_cast<size_t>(hv) * K);
    load_rows<IO, K>(ks_, static_cast<const IO*>(p.k), tok0, rows, static_cast<size_t>(p.H) * K, static_cast<size_t>(hk) * K);
    if (tid < C) bs[tid] = tid < rows ? p.beta[(tok0 + tid) * p.HV + hv] : 0.f;
    __syncthreads();
    cumsum_log2<K, LK>(gs);
    __syncthreads();
    if (tid < K) gl2[tid] = gs[(C - 1) * LK + tid];
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = tid + NT * u, i = c >> 4, d8 = (c & 15) << 3;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = ks_[i * LK + d8 + e] * ex2(gl2[d8 + e] - gs[i * LK + d8 + e]);
      uint4 hi, lo;
      split8(x, hi, lo);
      const uint32_t o = (d8 >> 6) * 8192u + sw_chunk(i, d8);
      *reinterpret_cast<uint4*>(sm + gvt::RKR + o) = hi;
      *reinterpret_cast<uint4*>(sm + gvt::RKR + 16384 + o) = lo;
    }
    __syncthreads();  // the scratch is read before h and D overwrite it
  }
  // 2. W and do split K-major; h and D split K-major (and dgl = e^{gl} sum_v h D); the
  //    addends -U^T and E^T into TMEM
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = tid + NT * u, i = c >> 4, c8 = (c & 15) << 3;
    const uint32_t o = (c8 >> 6) * 8192u + sw_chunk(i, c8);
    float x[8];
    const float4 a = *reinterpret_cast<const float4*>(slot + S::W + i * K + c8);
    const float4 b = *reinterpret_cast<const float4*>(slot + S::W + i * K + c8 + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    uint4 hi, lo;
    split8(x, hi, lo);
    *reinterpret_cast<uint4*>(sm + gvt::RW + o) = hi;
    *reinterpret_cast<uint4*>(sm + gvt::RW + 16384 + o) = lo;
    float4 da = make_float4(0.f, 0.f, 0.f, 0.f), db = da;
    if (i < rows) {
      da = load4(dop + static_cast<size_t>(tok0 + i) * vrow + vcol + c8);
      db = load4(dop + static_cast<size_t>(tok0 + i) * vrow + vcol + c8 + 4);
    }
    x[0] = da.x; x[1] = da.y; x[2] = da.z; x[3] = da.w; x[4] = db.x; x[5] = db.y; x[6] = db.z; x[7] = db.w;
    split8(x, hi, lo);
    *reinterpret_cast<uint4*>(sm + gvt::RDO + o) = hi;
    *reinterpret_cast<uint4*>(sm + gvt::RDO + 16384 + o) = lo;
  }
#pragma unroll 2
  for (int u = 0; u < 8; ++u) {
    const int c = tid + NT * u, d = c >> 4, v8 = (c & 15) << 3;
    const uint32_t o = (v8 >> 6) * 16384u + sw_chunk(d, v8);
    const float* hs = slot + S::RH + kv_off<K>(d, v8);
    const float* ds = slot + S::BD + kv_off<K>(d, v8);
    float xh[8], xd[8];
    const float4 h0 = *reinterpret_cast<const float4*>(hs), h1 = *reinterpret_cast<const float4*>(hs + 4);
    const float4 d0 = *reinterpret_cast<const float4*>(ds), d1 = *reinterpret_cast<const float4*>(ds + 4);
    xh[0] = h0.x; xh[1] = h0.y; xh[2] = h0.z; xh[3] = h0.w; xh[4] = h1.x; xh[5] = h1.y; xh[6] = h1.z; xh[7] = h1.w;
    xd[0] = d0.x; xd[1] = d0.y; xd[2] = d0.z; xd[3] = d0.w; xd[4] = d1.x; xd[5] = d1.y; xd[6] = d1.z; xd[7] = d1.w;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) dot = fmaf(xh[e], xd[e], dot);
#pragma unroll
    for (int o2 = 8; o2 >= 1; o2 >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o2);  // the row's 16 threads
    if ((tid & 15) == 0) slot[S::DGL + d] = ex2(gl2[d]) * dot;
    uint4 hi, lo;
    split8(xh, hi, lo);
    *reinterpret_cast<uint4*>(sm + gvt::RH + o) = hi;
    *reinterpret_cast<uint4*>(sm + gvt::RH + 32768 + o) = lo;
    split8(xd, hi, lo);
    *reinterpret_cast<uint4*>(sm + gvt::RD + o) = hi;
    *reinterpret_cast<uint4*>(sm + gvt::RD + 32768 + o) = lo;
  }
  {
    float a[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) a[j] = -slot[S::U + (hcol + j) * V + row];
    tmem_st32(tl, a);
#pragma unroll
    for (int j = 0; j < 32; ++j) a[j] = slot[S::E + (hcol + j) * V + row];
    tmem_st32(tl + 64, a);
    tmem_st_wait();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t id_ab = idesc_f16kind(128, 64) | IDESC_A_MN_MAJOR;  // A MN-major, B K-major
    constexpr uint32_t id_kk = idesc_f16kind(128, 64);                      // both K-major
    // -v_new^T (onto -U^T): A = h^T (MN-major view of h), B = W (K-major)
    issue_split(tmem, [&](int k) { return sdesc(sb + gvt::RH + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RH + 32768 + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc_sw128(sb + gvt::RW + (k >> 2) * 8192 + (k & 3) * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RW + 16384 + (k >> 2) * 8192 + (k & 3) * 32); }, id_ab, 8, true);
    // dv_new^T (onto E^T): A = D^T, B = kr
    issue_split(tmem + 64, [&](int k) { return sdesc(sb + gvt::RD + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RD + 32768 + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc_sw128(sb + gvt::RKR + (k >> 2) * 8192 + (k & 3) * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RKR + 16384 + (k >> 2) * 8192 + (k & 3) * 32); }, id_ab, 8, true);
    // DH^T: A = h (K-major), B = do (K-major)
    issue_split(tmem + 128, [&](int k) { return sdesc_sw128(sb + gvt::RH + (k >> 2) * 16384 + (k & 3) * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RH + 32768 + (k >> 2) * 16384 + (k & 3) * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RDO + (k >> 2) * 8192 + (k & 3) * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RDO + 16384 + (k >> 2) * 8192 + (k & 3) * 32); }, id_kk, 8, false);
    umma_commit(mbar);
  }
  wait_products();
  // 3. v_new^T and dv_new^T split as MN-major B tiles (K-rows = value columns) over W and kr;
  //    DH to the slot
  {
    float x[32];
    tmem_ld32(tl, x);
    tmem_ld_wait();
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = -x[8 * j8 + e];
      uint4 hi, lo;
      split8(y, hi, lo);
      const uint32_t o = sw_chunk(row, hcol + 8 * j8);
      *reinterpret_cast<uint4*>(sm + gvt::RW + o) = hi;
      *reinterpret_cast<uint4*>(sm + gvt::RW + 16384 + o) = lo;
    }
    tmem_ld32(tl + 64, x);
    tmem_ld_wait();
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = x[8 * j8 + e];
      uint4 hi, lo;
      split8(y, hi, lo);
      const uint32_t o = sw_chunk(row, hcol + 8 * j8);
      *reinterpret_cast<uint4*>(sm + gvt::RKR + o) = hi;
      *reinterpret_cast<uint4*>(sm + gvt::RKR + 16384 + o) = lo;
    }
    tmem_ld32(tl + 128, x);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) slot[S::DH + (hcol + j) * K + row] = x[j];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t id_kb = idesc_f16kind(128, 64) | IDESC_B_MN_MAJOR;  // A K-major, B MN-major
    // -dW^T: A = h, B = dv_new^T
    issue_split(tmem + 192, [&](int k) { return sdesc_sw128(sb + gvt::RH + (k >> 2) * 16384 + (k & 3) * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RH + 32768 + (k >> 2) * 16384 + (k & 3) * 32); },
                [&](int k) { return sdesc(sb + gvt::RKR + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RKR + 16384 + k * 2048, 16384, 1024, 2); }, id_kb, 8, false);
    // dkr^T: A = D, B = v_new^T
    issue_split(tmem + 256, [&](int k) { return sdesc_sw128(sb + gvt::RD + (k >> 2) * 16384 + (k & 3) * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RD + 32768 + (k >> 2) * 16384 + (k & 3) * 32); },
                [&](int k) { return sdesc(sb + gvt::RW + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RW + 16384 + k * 2048, 16384, 1024, 2); }, id_kb, 8, false);
    umma_commit(mbar);
  }
  wait_products();
  // 4. dW, dkr to the slot; over h and D: [do^T | dv_new^T] and [v_new^T | v^T] (two 64-wide
  //    atoms each, 16 KB apart); T Diag(beta) split as an MN-major B over do
  {
    float x[32];
    tmem_ld32(tl + 192, x);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) slot[S::DW + (hcol + j) * K + row] = -x[j];
    tmem_ld32(tl + 256, x);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) slot[S::DKR + (hcol + j) * K + row] = x[j];
    tmem_ld32(tl + 64, x);  // dv_new^T again
    tmem_ld_wait();
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = x[8 * j8 + e];
      uint4 hi, lo;
      split8(y, hi, lo);
      const uint32_t o = sw_chunk(row, hcol + 8 * j8);
      *reinterpret_cast<uint4*>(sm + gvt::RH + 16384 + o) = hi;
      *reinterpret_cast<uint4*>(sm + gvt::RH + 49152 + o) = lo;
    }
    tmem_ld32(tl, x);  // -v_new^T again
    tmem_ld_wait();
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = -x[8 * j8 + e];
      uint4 hi, lo;
      split8(y, hi, lo);
      const uint32_t o = sw_chunk(row, hcol + 8 * j8);
      *reinterpret_cast<uint4*>(sm + gvt::RD + o) = hi;
      *reinterpret_cast<uint4*>(sm + gvt::RD + 32768 + o) = lo;
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {  // do^T and v^T: K-row = value column, 8 chunk rows per chunk
    const int c = tid + NT * u, vv = c >> 3, i8 = (c & 7) << 3;
    float xo[8], xv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const bool ok = i8 + e < rows;
      const size_t at = static_cast<size_t>(tok0 + i8 + e) * vrow + vcol + vv;
      xo[e] = ok ? load1(dop + at) : 0.f;
      xv[e] = ok ? load1(vp + at) : 0.f;
    }
    const uint32_t o = sw_chunk(vv, i8);
    uint4 hi, lo;
    split8(xo, hi, lo);
    *reinterpret_cast<uint4*>(sm + gvt::RH + o) = hi;
    *reinterpret_cast<uint4*>(sm + gvt::RH + 32768 + o) = lo;
    split8(xv, hi, lo);
    *reinterpret_cast<uint4*>(sm + gvt::RD + 16384 + o) = hi;
    *reinterpret_cast<uint4*>(sm + gvt::RD + 49152 + o) = lo;
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {  // T Diag(beta): K-row = chunk row i, columns j
    const int c = tid + NT * u, i = c >> 3, j8 = (c & 7) << 3;
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = slot[S::T + i * C + j8 + e] * bs[j8 + e];
    uint4 hi, lo;
    split8(x, hi, lo);
    const uint32_t o = sw_chunk(i, j8);
    *reinterpret_cast<uint4*>(sm + gvt::RDO + o) = hi;
    *reinterpret_cast<uint4*>(sm + gvt::RDO + 8192 + o) = lo;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    constexpr uint32_t id_mm = idesc_f16kind(128, 128) | IDESC_A_MN_MAJOR | IDESC_B_MN_MAJOR;
    constexpr uint32_t id_kb = idesc_f16kind(128, 64) | IDESC_B_MN_MAJOR;
    // [do; dv_new] [v_new; v]^T
    issue_split(tmem + 320, [&](int k) { return sdesc(sb + gvt::RH + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RH + 32768 + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RD + k * 2048, 16384, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RD + 32768 + k * 2048, 16384, 1024, 2); }, id_mm, 8, false);
    // dv^T: A = dv_new^T (K-major view of its atom), B = T Diag(beta)
    issue_split(tmem + 448, [&](int k) { return sdesc_sw128(sb + gvt::RH + 16384 + k * 32); },
                [&](int k) { return sdesc_sw128(sb + gvt::RH + 49152 + k * 32); },
                [&](int k) { return sdesc(sb + gvt::RDO + k * 2048, 8192, 1024, 2); },
                [&](int k) { return sdesc(sb + gvt::RDO + 8192 + k * 2048, 8192, 1024, 2); }, id_kb, 4, false);
    umma_commit(mbar);
  }
  wait_products();
  // 5. dAqk (rows 0-63, columns 0-63) and dAv (rows 64-127, columns 64-127), lower
  //    triangles; dv
  {
    float x[32];
    const bool first = row < 64;
    tmem_ld32(tl + 320 + (first ? 0 : 64), x);
    tmem_ld_wait();
    const int i = first ? row : row - 64;
    float* dst = slot + (first ? S::DAQK : S::DAV) + i * C + hcol;
#pragma unroll
    for (int j = 0; j < 32; ++j) dst[j] = hcol + j <= i ? x[j] : 0.f;
    tmem_ld32(tl + 448, x);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (hcol + j < rows) p.dv[(static_cast<size_t>(tok0 + hcol + j) * p.HV + hv) * V + row] = x[j];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------- C x C stage --
template <int K>
struct GcSmem {
  static constexpr int LK = K + 4;
  static constexpr int B0 = 0, B1 = C * LK, XT = 2 * C * LK, XA = XT + C * LC, XY = XA + C * LC, XM = XY + C * LC,
                       XK = XM + C * LC, BS = XK + C * LC, DBC = BS + C, FLOATS = DBC + C;
};
template <typename IO, int K, int V>
__global__ void __launch_bounds__(NT, 1) grad_cc_kernel(Params p) {
  using S = Slot<K, V>;
  using L = GcSmem<K>;
  constexpr int LK = L::LK;
  extern __shared__ __align__(16) float sm[];
  float *B0 = sm + L::B0, *B1 = sm + L::B1, *XT = sm + L::XT, *XA = sm + L::XA, *XY = sm + L::XY, *XM = sm + L::XM,
        *XK = sm + L::XK, *bs = sm + L::BS, *dbc = sm + L::DBC;
  int seq, m, rows;
  long tok0;
  const int f = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
  if (!find_chunk(p, f, seq, m, tok0, rows)) return;
  const int hk = hv / (p.HV / p.H);
  float* slot = p.ws + (static_cast<size_t>(f) * p.HV + hv) * p.slot_floats;
  const auto lower = [](int m0, int n0) { return n0 <= m0 + 16; };

  load_rows<float, K>(B0, p.g, tok0, rows, static_cast<size_t>(p.HV) * K, static_cast<size_t>(hv) * K);
  load_rows<IO, K>(B1, static_cast<const IO*>(p.k), tok0, rows, static_cast<size_t>(p.H) * K, static_cast<size_t>(hk) * K);
  copy_in<C, LC>(XT, slot + S::T);
  copy_in<C, LC>(XA, slot + S::DAV);
  copy_in<C, LC>(XK, slot + S::KK);
  if (tid < C) bs[tid] = tid < rows ? p.beta[(tok0 + tid) * p.HV + hv] : 0.f;
  __syncthreads();
  cumsum_log2<K, LK>(B0);
  __syncthreads();
  for (int idx = tid; idx < C * K; idx += NT) {  // kd = k e^{gc}
    const int i = idx / K, d = idx - i * K;
    B0[i * LK + d] = B1[i * LK + d] * ex2(B0[i * LK + d]);
  }
  __syncthreads();
  copy_in<K, LK>(B1, slot + S::DW);
  __syncthreads();
  // dA = dW kd^T + dAv (lower, diagonal included), in place of dAv
  cta_gemm<C, C, 2, 2>([&](int i, int d, int) { return B1[i * LK + d]; }, [&](int d, int j, int) { return B0[j * LK + d]; }, lower,
                    [](int, int) { return make_int2(0, K); }, [&](int r, int c) { return XA[r * LC + c]; },
                    [&](int r, int c, float x0, float x1) {
                      XA[r * LC + c] = c <= r ? x0 : 0.f;
                      XA[r * LC + c + 1] = c + 1 <= r ? x1 : 0.f;
                    });
  __syncthreads();
  if (tid < C) {  // dbeta_j from A = T Diag(beta): sum_i T_ij dA_ij
    float s = 0.f;
    for (int i = tid; i < C; ++i) s = fmaf(XT[i * LC + tid], XA[i * LC + tid], s);
    dbc[tid] = s;
  }
  // Y = dA A^T (lower tiles): Y_aj = sum_{b <= j} dA_ab T_jb beta_b
  cta_gemm<C, C, 2, 2>([&](int a, int b, int) { return XA[a * LC + b]; }, [&](int b, int j, int) { return XT[j * LC + b] * bs[b]; },
                    lower, [](int, int n0) { return make_int2(0, n0 + 16); }, [](int, int) { return 0.f; },
                    [&](int r, int c, float x0, float x1) {
                      XY[r * LC + c] = x0;
                      XY[r * LC + c + 1] = x1;
                    });
  __syncthreads();
  // dM = -strict_tril(T^T Y): dM_ij = -sum_{a >= i} T_ai Y_aj
  cta_gemm<C, C, 2, 2>([&](int i, int a, int) { return XT[a * LC + i]; }, [&](int a, int j, int) { return XY[a * LC + j]; }, lower,
                    [](int m0, int) { return make_int2(m0, C); }, [](int, int) { return 0.f; },
                    [&](int r, int c, float x0, float x1) {
                      XM[r * LC + c] = c < r ? -x0 : 0.f;
                      XM[r * LC + c + 1] = c + 1 < r ? -x1 : 0.f;
                    });
  __syncthreads();
  if (tid < C) {  // dbeta_i from M = Diag(beta) KKd: sum_j dM_ij KKd_ij
    float s = dbc[tid];
    for (int j = 0; j < tid; ++j) s = fmaf(XM[tid * LC + j], XK[tid * LC + j], s);
    if (tid < rows) p.dbeta[(tok0 + tid) * p.HV + hv] = s;
  }
  for (int idx = tid; idx < C * C; idx += NT) {
    const int r = idx >> 6, c = idx & 63;
    slot[S::DMB + idx] = bs[r] * XM[r * LC + c];
  }
}

// ------------------------------------------------------------ key gradients --
constexpr int DK = 64;  // key dims per grad_k CTA
constexpr int LD = DK + 4;
struct GkSmem {
  static constexpr int GC = 0, LKT = GC + C * LD, LQT = LKT + C * LD, RT = LQT + C * LD, KR = RT + C * LD,
                       QR = KR + C * LD, DW = QR + C * LD, DKA = DW + C * LD, DGA = DKA + C * LD, XT = DGA + C * LD,
                       XQ = XT + C * LC, XM = XQ + C * LC, REF = XM + C * LC, BS = REF + 8 * DK, FLOATS = BS + C;
};
template <typename IO, int K, int V>
__global__ void __launch_bounds__(NT, 1) grad_k_kernel(Params p) {
  using S = Slot<K, V>;
  using L = GkSmem;
  extern __shared__ __align__(16) float sm[];
  float *GC = sm + L::GC, *LKt = sm + L::LKT, *LQt = sm + L::LQT, *RT = sm + L::RT, *KR = sm + L::KR, *QR = sm + L::QR,
        *DWs = sm + L::DW, *DKA = sm + L::DKA, *DGA = sm + L::DGA, *XT = sm + L::XT, *XQ = sm + L::XQ, *XM = sm + L::XM,
        *refs = sm + L::REF, *bs = sm + L::BS;
  int seq, m, rows;
  long tok0;
  const int f = blockIdx.x, hv = blockIdx.y, d0 = blockIdx.z * DK, tid = threadIdx.x, warp = tid >> 5;
  if (!find_chunk(p, f, seq, m, tok0, rows)) return;
  const int hk = hv / (p.HV / p.H);
  const float* slot = p.ws + (static_cast<size_t>(f) * p.HV + hv) * p.slot_floats;
  const size_t qk_row = static_cast<size_t>(p.H) * K, qk_col = static_cast<size_t>(hk) * K + d0;

  {  // the fp32 tiles by cp.async, all in flight together (g rows past the chunk are zero)
    const float* gp = p.g + static_cast<size_t>(tok0) * p.HV * K + static_cast<size_t>(hv) * K + d0;
    for (int idx = tid; idx < C * (DK / 4); idx += NT) {
      const int r = idx / (DK / 4), c4 = (idx - r * (DK / 4)) * 4;
      if (r < rows)
        cp_async16(GC + r * LD + c4, gp + static_cast<size_t>(r) * p.HV * K + c4);
      else
        *reinterpret_cast<float4*>(GC + r * LD + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
      cp_async16(DWs + r * LD + c4, slot + S::DW + static_cast<size_t>(r) * K + d0 + c4);
    }
    for (int idx = tid; idx < C * (C / 4); idx += NT) {
      const int r = idx / (C / 4), c4 = (idx - r * (C / 4)) * 4;
      cp_async16(XT + r * LC + c4, slot + S::T + r * C + c4);
      cp_async16(XQ + r * LC + c4, slot + S::DAQK + r * C + c4);
      cp_async16(XM + r * LC + c4, slot + S::DMB + r * C + c4);
    }
    cp_async_commit();
  }
  load_rows<IO, DK>(KR, static_cast<const IO*>(p.k), tok0, rows, qk_row, qk_col);
  load_rows<IO, DK>(QR, static_cast<const IO*>(p.q), tok0, rows, qk_row, qk_col);
  if (tid < C) bs[tid] = tid < rows ? p.beta[(tok0 + tid) * p.HV + hv] : 0.f;
  cp_async_wait<0>();
  __syncthreads();
  // tables: Lk, Lq from copies of the raw rows (the raw rows stay for the final pass)
  for (int idx = tid; idx < C * DK; idx += NT) {
    const int i = idx / DK, d = idx - i * DK;
    LKt[i * LD + d] = KR[i * LD + d];
    LQt[i * LD + d] = QR[i * LD + d];
  }
  __syncthreads();
  make_tables<DK, LD>(LKt, LQt, GC, RT, refs, p.scale);
  __syncthreads();
  const int m0 = 16 * (warp >> 1), n0 = 32 * (warp & 1), bi0 = m0 >> 4;  // one 16 x 32 tile of C x 64 per warp
  const int lane = tid & 31, g = lane >> 2, t = lane & 3;
  // 1. dkd = A^T dW -> dk_acc = e^{gc} dkd, dgc_acc = k e^{gc} dkd
  {
    float acc[4][4];
    tile_init<4>(acc, [](int, int) { return 0.f; }, m0, n0);
    tile_mma<4>(acc, [&](int j, int i, int) { return XT[i * LC + j] * bs[j]; }, [&](int i, int d, int) { return DWs[i * LD + d]; },
                m0, n0, m0, C);
    tile_epi<4>(acc, [&](int r, int c, float x0, float x1) {
      const float y0 = ex2(GC[r * LD + c]) * x0, y1 = ex2(GC[r * LD + c + 1]) * x1;
      DKA[r * LD + c] = y0;
      DKA[r * LD + c + 1] = y1;
      DGA[r * LD + c] = KR[r * LD + c] * y0;
      DGA[r * LD + c + 1] = KR[r * LD + c + 1] * y1;
    }, m0, n0);
  }
  // 2. row side: X_i = sum_j P_ij k_j e^{gc_i - gc_j} for P = dMb (dk) and dAqk (dq), by
  //    column blocks with the accumulator rescaled between them
  {
    float ak[4][4], aq[4][4];
    tile_init<4>(ak, [](int, int) { return 0.f; }, m0, n0);
    tile_init<4>(aq, [](int, int) { return 0.f; }, m0, n0);
    for (int bj = 0; bj <= bi0; ++bj) {
      if (bj > 0) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = n0 + 8 * nt + 2 * t + (e & 1);
            const float s = ex2(refs[(4 + bj) * DK + d] - refs[(3 + bj) * DK + d]);
            ak[nt][e] *= s;
            aq[nt][e] *= s;
          }
      }
      const auto fb = [&](int j, int d, int) { return RT[j * LD + d]; };
      tile_mma<4>(ak, [&](int i, int j, int) { return XM[i * LC + j]; }, fb, m0, n0, 16 * bj, 16 * bj + 16);
      tile_mma<4>(aq, [&](int i, int j, int) { return XQ[i * LC + j]; }, fb, m0, n0, 16 * bj, 16 * bj + 16);
    }
    const float scale = p.scale;
    float* dqp = p.dq + static_cast<size_t>(tok0) * qk_row + qk_col;
    const float* dh = slot + S::DH + d0;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + g + 8 * (e >> 1), d = n0 + 8 * nt + 2 * t + (e & 1);
        const float x = GC[r * LD + d];
        const float fr = ex2(x - refs[(4 + bi0) * DK + d]);
        const float dkr = ak[nt][e] * fr;
        DKA[r * LD + d] += dkr;
        DGA[r * LD + d] += KR[r * LD + d] * dkr;
        const float dq = scale * (ex2(x) * dh[static_cast<size_t>(r) * K + d] + aq[nt][e] * fr);
        DGA[r * LD + d] += QR[r * LD + d] * dq;
        if (r < rows) atomicAdd(dqp + static_cast<size_t>(r) * qk_row + d, dq);
      }
  }
  // 3. column side: Y_j = sum_i (dAqk_ij scale q_i + dMb_ij k_i) e^{gc_i - gc_j}, by row
  //    blocks from the last, rescaled between them
  {
    float ac[4][4];
    tile_init<4>(ac, [](int, int) { return 0.f; }, m0, n0);
    for (int bi = 3; bi >= bi0; --bi) {
      if (bi < 3) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = n0 + 8 * nt + 2 * t + (e & 1);
            ac[nt][e] *= ex2(refs[(bi + 1) * DK + d] - refs[bi * DK + d]);
          }
      }
      tile_mma<4>(ac, [&](int j, int i, int) { return XQ[i * LC + j]; }, [&](int i, int d, int) { return LQt[i * LD + d]; }, m0, n0,
                  16 * bi, 16 * bi + 16);
      tile_mma<4>(ac, [&](int j, int i, int) { return XM[i * LC + j]; }, [&](int i, int d, int) { return LKt[i * LD + d]; }, m0, n0,
                  16 * bi, 16 * bi + 16);
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + g + 8 * (e >> 1), d = n0 + 8 * nt + 2 * t + (e & 1);
        const float y = ac[nt][e] * ex2(refs[bi0 * DK + d] - GC[r * LD + d]);
        DKA[r * LD + d] += y;
        DGA[r * LD + d] -= KR[r * LD + d] * y;
      }
  }
  // 4. dk_e^{gl-gc} = dkr e^{gl - gc}; dk out; dgc; dg = reverse cumulative sum
  {
    const float* dkr = slot + S::DKR + d0;
    float* dkp = p.dk + static_cast<size_t>(tok0) * qk_row + qk_col;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = m0 + g + 8 * (e >> 1), d = n0 + 8 * nt + 2 * t + (e & 1);
        const float x = dkr[static_cast<size_t>(r) * K + d] * ex2(refs[7 * DK + d] - GC[r * LD + d]);
        const float dkv = DKA[r * LD + d] + x;
        DGA[r * LD + d] -= KR[r * LD + d] * x;
        DKA[r * LD + d] = KR[r * LD + d] * x;  // (now k dk_e^{gl-gc}, summed over rows below)
        if (r < rows) atomicAdd(dkp + static_cast<size_t>(r) * qk_row + d, dkv);
      }
  }
  __syncthreads();
  {  // four threads per key dim, 16 rows each: the column sum of k dk_e^{gl-gc} and the
     // segment sums of dgc (in refs, free now), then each segment's reverse cumulative sum
    const int col = tid & (DK - 1), part = tid / DK;
    float sk = 0.f, sg = 0.f;
#pragma unroll
    for (int i = 16 * part; i < 16 * part + 16; ++i) {
      sk += DKA[i * LD + col];
      sg += DGA[i * LD + col];
    }
    refs[part * DK + col] = sk;
    refs[4 * DK + part * DK + col] = sg;
    __syncthreads();
    float s = slot[S::DGL + d0 + col];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      s += refs[q * DK + col];
      if (q > part) s += refs[4 * DK + q * DK + col];
    }
    float* dgp = p.dg + static_cast<size_t>(tok0) * p.HV * K + static_cast<size_t>(hv) * K + d0 + col;
#pragma unroll
    for (int i = 16 * part + 15; i >= 16 * part; --i) {
      s += DGA[i * LD + col];
      if (i < rows) dgp[static_cast<size_t>(i) * p.HV * K] = s;
    }
  }
}

template <typename IO, int K, int V>
cudaError_t launch_kv(const Params& p, int chunks, cudaStream_t st) {
  const size_t s_prep = PrepSmem<K, V>::BYTES, s_chain = K == 128 ? tcc::SMEM : ChainSmem<K>::FLOATS * 4,
               s_gv = GvSmem<K, V>::FLOATS * 4,
               s_gc = GcSmem<K>::FLOATS * 4, s_gk = GkSmem::FLOATS * 4;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(prep_kernel<IO, K, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_prep)) != cudaSuccess ||
      (e = K == 128 ? cudaFuncSetAttribute(chain_tc_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_chain)
                    : cudaFuncSetAttribute(chain_kernel<K, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_chain)) !=
          cudaSuccess ||
      (e = (K == 128 && V == 128)
               ? cudaFuncSetAttribute(grad_v_tc_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gvt::SMEM)
               : cudaFuncSetAttribute(grad_v_kernel<IO, K, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_gv)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(grad_cc_kernel<IO, K, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_gc)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(grad_k_kernel<IO, K, V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_gk)) != cudaSuccess)
    return e;
  if (chunks > 0) {
    prep_kernel<IO, K, V><<<dim3(chunks, p.HV), NT, s_prep, st>>>(p);
  }
  if (K == 128)
    chain_tc_kernel<V><<<dim3(V < VS ? 1 : V / VS, p.HV, 2 * p.num_seqs), NT, s_chain, st>>>(p);
  else
    chain_kernel<K, V><<<dim3(V < VS ? 1 : V / VS, p.HV, 2 * p.num_seqs), NT, s_chain, st>>>(p);
  if (chunks > 0) {
    if (K == 128 && V == 128)
      grad_v_tc_kernel<IO><<<dim3(chunks, p.HV), NT, gvt::SMEM, st>>>(p);
    else
      grad_v_kernel<IO, K, V><<<dim3(chunks, p.HV), NT, s_gv, st>>>(p);
    grad_cc_kernel<IO, K, V><<<dim3(chunks, p.HV), NT, s_gc, st>>>(p);
    grad_k_kernel<IO, K, V><<<dim3(chunks, p.HV, K / DK), NT, s_gk, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace cbwd

// Flat chunk slots the chunk-form backward needs: every chunk of every sequence (a bound
// when the lengths are on the device: T / 64 + one partial chunk per sequence).
size_t backward_chunk_slots(long T, int num_seqs_or_B, bool varlen, int HV) {
  const long nc = (T + cbwd::C - 1) / cbwd::C;
  const long chunks = varlen ? nc + num_seqs_or_B : nc * num_seqs_or_B;
  return static_cast<size_t>(chunks) * HV;
}
size_t backward_chunk_slot_floats(int K, int V) {
  if (K == 128 && V == 128) return cbwd::Slot<128, 128>::FLOATS;
  if (K == 128 && V == 64) return cbwd::Slot<128, 64>::FLOATS;
  if (K == 64 && V == 128) return cbwd::Slot<64, 128>::FLOATS;
  return cbwd::Slot<64, 64>::FLOATS;
}

cudaError_t launch_backward_chunk(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  const float* s0, const int32_t* cu, const void* d_out, const float* d_fin, float* dq,
                                  float* dk, float* dv, float* dg, float* dbeta, float* ds0, float* ws,
                                  uint32_t* status, unsigned long long wait_ns, float scale, int T, int H, int HV,
                                  int K, int V, int num_seqs, bool bf16, cudaStream_t stream) {
  const int nc = (T + cbwd::C - 1) / cbwd::C;
  const int chunks = cu ? nc + num_seqs : nc * num_seqs;
  cbwd::Params p{q,  k,  v,  g,     beta,   s0,  cu, d_out, d_fin, dq, dk, dv, dg, dbeta, ds0, ws, status,
                 backward_chunk_slot_floats(K, V), wait_ns, scale, T, H, HV, num_seqs, nc};
  if (bf16) {
    if (K == 128 && V == 128) return cbwd::launch_kv<__nv_bfloat16, 128, 128>(p, chunks, stream);
    if (K == 128 && V == 64) return cbwd::launch_kv<__nv_bfloat16, 128, 64>(p, chunks, stream);
    if (K == 64 && V == 128) return cbwd::launch_kv<__nv_bfloat16, 64, 128>(p, chunks, stream);
    return cbwd::launch_kv<__nv_bfloat16, 64, 64>(p, chunks, stream);
  }
  if (K == 128 && V == 128) return cbwd::launch_kv<float, 128, 128>(p, chunks, stream);
  if (K == 128 && V == 64) return cbwd::launch_kv<float, 128, 64>(p, chunks, stream);
  if (K == 64 && V == 128) return cbwd::launch_kv<float, 64, 128>(p, chunks, stream);
  return cbwd::launch_kv<float, 64, 64>(p, chunks, stream);
}

}  // namespace kda
