// kda_backward.cu -- gradients of the forward with respect to q, k, v, g, beta and
// the initial state, by reverse mode through the token recurrence, on CUDA cores in
// fp32.
//
// For the loss sum_t <do_t, o_t> + <dS_final, S_final>, going back from the last token,
// with Sp the state before token t, P = Diag(e^{g_t}) Sp, u = P^T k, r = v - u and
// S = P + beta k r^T (the recurrence of page "手撕KDA", section "1 Naive"):
//     dq_t = scale S do_t;  dS += scale q_t do_t^T
//     kd = dS^T k;  dbeta_t = r . kd;  dr = beta kd;  dv_t = dr
//     dk_t = beta dS r - P dr;  dP = dS - k dr^T;  dg_t,i = sum_j dP_ij P_ij;  dS = Diag(e^{g_t}) dP
// and dS after the first token is the initial state's gradient.  (The pages' backward,
// "手撕KDA" sections 2 and 4, works on the chunked form; this is the same derivative
// taken through the recurrence it evaluates.)
//
// The state recurrence and its reverse are independent across value columns; only dq,
// dk, dg and dbeta sum over them.  So each (sequence, value head) is split into V / 32
// slices of 32 value columns, one CTA each: 256 threads, each holding 4 adjacent columns
// of K / 32 state rows.  The states the reverse sweep needs are recomputed: a forward
// sweep stores the fp32 state slice entering every 64-token chunk in the workspace,
// then, chunk by chunk from the last, the chunk's 64 token states are recomputed into
// the workspace and swept in reverse.  Reductions over K go through shared memory,
// reductions over a slice's columns are warp shuffles among the row's 8 lanes (a
// halving reduce-scatter: one row sum per lane pair); the slices' partial dq, dk, dg
// and dbeta (and those of the value heads sharing a key head, for dq and dk) meet in
// fp32 atomics on outputs the launcher zeroes first.
#include "kda_common.cuh"

namespace kda {
namespace bwd {

constexpr int NT = 256;
constexpr int CH = 64;  // tokens per checkpoint
constexpr int VS = 32;  // value columns per CTA

struct Params {
  const void* q;       // [tokens, H, K]  io type
  const void* k;
  const void* v;       // [tokens, HV, V]
  const float* g;      // [tokens, HV, K]
  const float* beta;   // [tokens, HV]
  const float* s0;     // [NS, HV, K, V] or null
  const int32_t* cu;   // [NS + 1] or null
  const void* d_out;   // [tokens, HV, V]  io type
  const float* d_fin;  // [NS, HV, K, V] or null
  float* dq;           // [tokens, H, K]  fp32, accumulated
  float* dk;
  float* dv;           // [tokens, HV, V]
  float* dg;           // [tokens, HV, K]
  float* dbeta;        // [tokens, HV]
  float* ds0;          // [NS, HV, K, V] or null
  float* scratch;      // per unit: (max chunks + CH) x K x V fp32 (V / 32 slices of it)
  uint32_t* status;
  size_t unit_floats;  // floats of scratch per unit
  float scale;
  int T, H, HV, num_seqs;
};

__device__ __forceinline__ bool seq_bounds(const Params& p, int seq, long& tok0, int& len) {
  if (!p.cu) {
    tok0 = static_cast<long>(seq) * p.T;
    len = p.T;
    return true;
  }
  const int a = p.cu[seq], b = p.cu[seq + 1];
  if (a < 0 || b < a || b > p.T || (seq == 0 && a != 0) || (seq == p.num_seqs - 1 && b != p.T)) {
    atomicOr(p.status, kStatusBounds);
    tok0 = 0;
    len = 0;
    return false;
  }
  tok0 = a;
  len = b - a;
  return true;
}

// Sums over the L lanes of a row group of N values per lane (xor masks M, M/2, .. 1 with
// M = L / 2): while more than one value is left each step keeps half and sends half, so
// every lane ends with the full sum of one value, index `idx`.
template <int N, int M>
struct Halve {
  static __device__ __forceinline__ void run(float* v, int lane, int& idx) {
    if constexpr (N > 1) {
      const bool up = (lane & M) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[i + N / 2];
        const float keep = up ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, M);
      }
      if (up) idx += N / 2;
      if constexpr (M > 1) Halve<N / 2, M / 2>::run(v, lane, idx);
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], M);
      if constexpr (M > 1) Halve<1, M / 2>::run(v, lane, idx);
    }
  }
};
// lanes that hold a distinct sum after Halve<N, L/2> (the others repeat one of them)
template <int N, int L>
__device__ __forceinline__ bool halve_writer(int lane) {
  int plain = 0;  // masks of the steps that only added
  int n = N;
  for (int m = L / 2; m >= 1; m /= 2) {
    if (n > 1) n /= 2;
    else plain |= m;
  }
  return (lane & plain) == 0;
}

template <typename IO, int K, int V>
__global__ void __launch_bounds__(NT) recurrent_bwd_kernel(const Params p) {
  constexpr int TPR = VS / 4;   // threads across a state row of the slice
  constexpr int RG = NT / TPR;  // row groups
  constexpr int RPT = K / RG;   // rows per thread: rg + RG i
  constexpr int NSPLIT = V / VS;
  static_assert(RPT * RG == K && TPR == 8 && NSPLIT * VS == V && K + VS <= NT, "backward tiling");
  const int slice = blockIdx.x, hv = blockIdx.y, seq = blockIdx.z;
  const int v0 = VS * slice;
  const int tid = threadIdx.x, lane = tid & 31;
  const int cg = tid % TPR, rg = tid / TPR;
  const int hk = hv / (p.HV / p.H);
  const IO* q = static_cast<const IO*>(p.q);
  const IO* k = static_cast<const IO*>(p.k);
  const IO* v = static_cast<const IO*>(p.v);
  const IO* dout = static_cast<const IO*>(p.d_out);

  // token inputs, double-buffered by step parity: a step stages the next token into the
  // other buffer between the two barriers of one of its reductions over K
  __shared__ float s_q[2][K], s_k[2][K], s_e[2][K], s_v[2][VS], s_do[2][VS], s_b[2];
  constexpr int NW = NT / 32;
  __shared__ __align__(16) float red[NW][VS];
  __shared__ __align__(16) float col[VS];   // a reduced vector over the slice's columns (u, then kd)

  long tok0;
  int len;
  seq_bounds(p, seq, tok0, len);
  const int nch = (len + CH - 1) / CH;
  const size_t unit = static_cast<size_t>(seq) * p.HV + hv;
  const size_t state_col = unit * K * V + v0 + 4 * cg;  // this thread's columns in a [K][V] state
  float* ckpt = p.scratch + unit * p.unit_floats + slice * (p.unit_floats / NSPLIT);  // [nch][K][VS]
  float* toks = ckpt + static_cast<size_t>(nch > 0 ? nch : 1) * K * VS;              // [CH][K][VS]
  auto slot = [&](float* base, int i) { return base + static_cast<size_t>(rg + RG * i) * VS + 4 * cg; };

  // Token inputs (q, k, g; the slice of v and do; beta) are fetched into registers one
  // token ahead and staged into shared memory at the next step, so that no step waits
  // for its own global loads: fetch(t) issues the loads, stage() writes the values.
  float f0 = 0.f, f1 = 0.f, f2 = 0.f;
  auto fetch = [&](int t) {
    const size_t tok = static_cast<size_t>(tok0 + t);
    if (tid < K) {
      f0 = to_f32(q[(tok * p.H + hk) * K + tid]);
      f1 = to_f32(k[(tok * p.H + hk) * K + tid]);
      f2 = p.g[(tok * p.HV + hv) * K + tid];
    } else if (tid < K + VS) {
      f0 = to_f32(v[(tok * p.HV + hv) * V + v0 + (tid - K)]);
      f1 = to_f32(dout[(tok * p.HV + hv) * V + v0 + (tid - K)]);
    } else if (tid == NT - 1) {
      f0 = p.beta[tok * p.HV + hv];
    }
  };
  auto stage = [&](int b) {
    if (tid < K) {
      s_q[b][tid] = f0;
      s_k[b][tid] = f1;
      s_e[b][tid] = expf(f2);
    } else if (tid < K + VS) {
      s_v[b][tid - K] = f0;
      s_do[b][tid - K] = f1;
    } else if (tid == NT - 1) {
      s_b[b] = f0;
    }
  };
  // x^T k over all rows (of the token in buffer b) -> col[].  Between its two barriers
  // (every thread has finished the previous step after the first) the fetched token goes
  // into buffer sb (if sb >= 0) and token ft is fetched (if ft >= 0); the second barrier
  // makes the staged values visible.
  auto reduce_k = [&](const float4 (&x)[RPT], int b, int sb, int ft) {
    float4 pu = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float kd = s_k[b][rg + RG * i];
      pu.x = fmaf(kd, x[i].x, pu.x); pu.y = fmaf(kd, x[i].y, pu.y);
      pu.z = fmaf(kd, x[i].z, pu.z); pu.w = fmaf(kd, x[i].w, pu.w);
    }
    // the warp's four row groups (lanes 8 apart hold the same columns), then the warps
#pragma unroll
    for (int m = TPR; m < 32; m <<= 1) {
      pu.x += __shfl_xor_sync(0xFFFFFFFFu, pu.x, m);
      pu.y += __shfl_xor_sync(0xFFFFFFFFu, pu.y, m);
      pu.z += __shfl_xor_sync(0xFFFFFFFFu, pu.z, m);
      pu.w += __shfl_xor_sync(0xFFFFFFFFu, pu.w, m);
    }
    if (lane < TPR) *reinterpret_cast<float4*>(&red[tid >> 5][4 * cg]) = pu;
    __syncthreads();
    if (tid < VS) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) a += red[w][tid];
      col[tid] = a;
    }
    if (sb >= 0) {
      stage(sb);
      if (ft >= 0) fetch(ft);
    }
    __syncthreads();
  };
  // one forward step on the state held in s (token in buffer b)
  auto forward_step = [&](float4 (&s)[RPT], int b, int sb, int ft) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float e = s_e[b][rg + RG * i];
      s[i].x *= e; s[i].y *= e; s[i].z *= e; s[i].w *= e;
    }
    reduce_k(s, b, sb, ft);
    const float bt = s_b[b];
    const float4 br = make_float4(bt * (s_v[b][4 * cg] - col[4 * cg]), bt * (s_v[b][4 * cg + 1] - col[4 * cg + 1]),
                                  bt * (s_v[b][4 * cg + 2] - col[4 * cg + 2]), bt * (s_v[b][4 * cg + 3] - col[4 * cg + 3]));
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float kd = s_k[b][rg + RG * i];
      s[i].x = fmaf(kd, br.x, s[i].x); s[i].y = fmaf(kd, br.y, s[i].y);
      s[i].z = fmaf(kd, br.z, s[i].z); s[i].w = fmaf(kd, br.w, s[i].w);
    }
  };

  // ---- 1. forward sweep: the fp32 state entering every chunk ----
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    s[i] = p.s0 ? *reinterpret_cast<const float4*>(p.s0 + state_col + static_cast<size_t>(rg + RG * i) * V)
                : make_float4(0.f, 0.f, 0.f, 0.f);
  if (len > 0) {
    fetch(0);
    stage(0);
    if (len > 1) fetch(1);
  }
  __syncthreads();
  for (int t = 0; t < len; ++t) {
    if (t % CH == 0) {
#pragma unroll
      for (int i = 0; i < RPT; ++i) *reinterpret_cast<float4*>(slot(ckpt + static_cast<size_t>(t / CH) * K * VS, i)) = s[i];
    }
    const int b = t & 1;
    // token t + 1 into the other buffer, token t + 2 fetched
    forward_step(s, b, t + 1 < len ? (b ^ 1) : -1, t + 2 < len ? t + 2 : -1);
  }

  // ---- 2. reverse sweep, one chunk at a time ----
  float4 ds[RPT];  // the state's gradient
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    ds[i] = p.d_fin ? *reinterpret_cast<const float4*>(p.d_fin + state_col + static_cast<size_t>(rg + RG * i) * V)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  const bool writer = halve_writer<RPT, TPR>(lane);
  for (int n = nch - 1; n >= 0; --n) {
    const int t0 = n * CH, t1 = min(len, t0 + CH);
    // recompute the chunk's token states (the state before each token)
#pragma unroll
    for (int i = 0; i < RPT; ++i) s[i] = *reinterpret_cast<const float4*>(slot(ckpt + static_cast<size_t>(n) * K * VS, i));
    // (the previous sweep's readers of both buffers are done before anything is staged)
    __syncthreads();
    if (t0 + 1 < t1) {
      fetch(t0);
      stage(0);
      if (t0 + 2 < t1) fetch(t0 + 1);
    }
    __syncthreads();
    for (int t = t0; t < t1; ++t) {
#pragma unroll
      for (int i = 0; i < RPT; ++i) *reinterpret_cast<float4*>(slot(toks + static_cast<size_t>(t - t0) * K * VS, i)) = s[i];
      if (t + 1 == t1) break;  // the last token's successor is not needed
      const int b = (t - t0) & 1;
      forward_step(s, b, t + 2 < t1 ? (b ^ 1) : -1, t + 3 < t1 ? t + 2 : -1);
    }
    // reverse: the inputs and the token states are read one token ahead too (this thread
    // wrote the states above)
    __syncthreads();
    fetch(t1 - 1);
    stage(0);
    if (t1 - 1 > t0) fetch(t1 - 2);
    float4 Pn[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) Pn[i] = *reinterpret_cast<const float4*>(slot(toks + static_cast<size_t>(t1 - 1 - t0) * K * VS, i));
    __syncthreads();
    for (int t = t1 - 1; t >= t0; --t) {
      const int b = (t1 - 1 - t) & 1;
      float4 P[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) P[i] = Pn[i];
      if (t > t0) {
#pragma unroll
        for (int i = 0; i < RPT; ++i) Pn[i] = *reinterpret_cast<const float4*>(slot(toks + static_cast<size_t>(t - 1 - t0) * K * VS, i));
      }
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float e = s_e[b][rg + RG * i];
        P[i].x *= e; P[i].y *= e; P[i].z *= e; P[i].w *= e;
      }
      reduce_k(P, b, -1, -1);  // col = u
      const float bt = s_b[b], sc = p.scale;
      const float4 r = make_float4(s_v[b][4 * cg] - col[4 * cg], s_v[b][4 * cg + 1] - col[4 * cg + 1],
                                   s_v[b][4 * cg + 2] - col[4 * cg + 2], s_v[b][4 * cg + 3] - col[4 * cg + 3]);
      const float4 dov = *reinterpret_cast<const float4*>(&s_do[b][4 * cg]);
      // dq = scale (P + beta k r^T) do, per row; then dS += scale q do^T
      float acc[RPT];
      const float rdo = bt * (r.x * dov.x + r.y * dov.y + r.z * dov.z + r.w * dov.w);
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int d = rg + RG * i;
        acc[i] = P[i].x * dov.x + P[i].y * dov.y + P[i].z * dov.z + P[i].w * dov.w + s_k[b][d] * rdo;
        const float qs = sc * s_q[b][d];
        ds[i].x = fmaf(qs, dov.x, ds[i].x); ds[i].y = fmaf(qs, dov.y, ds[i].y);
        ds[i].z = fmaf(qs, dov.z, ds[i].z); ds[i].w = fmaf(qs, dov.w, ds[i].w);
      }
      const size_t tok = static_cast<size_t>(tok0 + t);
      {
        int idx = 0;
        Halve<RPT, TPR / 2>::run(acc, lane, idx);
        if (writer) atomicAdd(p.dq + (tok * p.H + hk) * K + rg + RG * idx, sc * acc[0]);
      }
      // kd = dS^T k (all rows) -> col;  dr = beta kd;  dbeta = r . kd.  (Every thread has read
      // col (u) before it reaches the first barrier inside, after which col is rewritten;
      // the token before goes into the other buffer between the two.)
      reduce_k(ds, b, t > t0 ? (b ^ 1) : -1, t - 1 > t0 ? t - 2 : -1);
      const float4 kdv = *reinterpret_cast<const float4*>(&col[4 * cg]);
      const float4 dr = make_float4(bt * kdv.x, bt * kdv.y, bt * kdv.z, bt * kdv.w);
      if (rg == 0) *reinterpret_cast<float4*>(p.dv + (tok * p.HV + hv) * V + v0 + 4 * cg) = dr;
      {  // dbeta: every row group holds the slice's columns of r and kd; row group 0's sum is kept
        float db = r.x * kdv.x + r.y * kdv.y + r.z * kdv.z + r.w * kdv.w;
#pragma unroll
        for (int m = TPR / 2; m >= 1; m >>= 1) db += __shfl_xor_sync(0xFFFFFFFFu, db, m);
        if (tid == 0) atomicAdd(p.dbeta + tok * p.HV + hv, db);
      }
      // dk = beta dS r - P dr;  dP = dS - k dr^T;  dg = sum_j dP P;  dS = Diag(e) dP
      float dkv[RPT], dgv[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int d = rg + RG * i;
        const float kd = s_k[b][d], e = s_e[b][d];
        dkv[i] = bt * (ds[i].x * r.x + ds[i].y * r.y + ds[i].z * r.z + ds[i].w * r.w) -
                 (P[i].x * dr.x + P[i].y * dr.y + P[i].z * dr.z + P[i].w * dr.w);
        float4 dp = make_float4(ds[i].x - kd * dr.x, ds[i].y - kd * dr.y, ds[i].z - kd * dr.z, ds[i].w - kd * dr.w);
        dgv[i] = dp.x * P[i].x + dp.y * P[i].y + dp.z * P[i].z + dp.w * P[i].w;
        ds[i] = make_float4(e * dp.x, e * dp.y, e * dp.z, e * dp.w);
      }
      {
        int idx = 0;
        Halve<RPT, TPR / 2>::run(dkv, lane, idx);
        if (writer) atomicAdd(p.dk + (tok * p.H + hk) * K + rg + RG * idx, dkv[0]);
      }
      {
        int idx = 0;
        Halve<RPT, TPR / 2>::run(dgv, lane, idx);
        if (writer) atomicAdd(p.dg + (tok * p.HV + hv) * K + rg + RG * idx, dgv[0]);
      }
    }
  }
  if (p.ds0) {
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      *reinterpret_cast<float4*>(p.ds0 + state_col + static_cast<size_t>(rg + RG * i) * V) = ds[i];
  }
}

template <typename IO>
cudaError_t launch_io(const Params& p, int K, int V, cudaStream_t stream) {
  const dim3 grid(V / VS, p.HV, p.num_seqs);
  if (K == 128 && V == 128) recurrent_bwd_kernel<IO, 128, 128><<<grid, NT, 0, stream>>>(p);
  else if (K == 128 && V == 64) recurrent_bwd_kernel<IO, 128, 64><<<grid, NT, 0, stream>>>(p);
  else if (K == 64 && V == 128) recurrent_bwd_kernel<IO, 64, 128><<<grid, NT, 0, stream>>>(p);
  else recurrent_bwd_kernel<IO, 64, 64><<<grid, NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bwd

// floats of backward scratch per (sequence, value head): the chunk checkpoints of the
// longest possible sequence plus one chunk of token states
size_t backward_unit_floats(long max_len, int K, int V) {
  const long nch = (max_len + bwd::CH - 1) / bwd::CH;
  return static_cast<size_t>((nch > 0 ? nch : 1) + bwd::CH) * K * V;
}

cudaError_t launch_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const float* s0, const int32_t* cu, const void* d_out, const float* d_fin, float* dq,
                            float* dk, float* dv, float* dg, float* dbeta, float* ds0, float* scratch,
                            size_t unit_floats, uint32_t* status, float scale, int T, int H, int HV, int K, int V,
                            int num_seqs, bool bf16, cudaStream_t stream) {
  bwd::Params p{q, k, v, g, beta, s0, cu, d_out, d_fin, dq, dk, dv, dg, dbeta, ds0, scratch, status, unit_floats,
                scale, T, H, HV, num_seqs};
  return bf16 ? bwd::launch_io<__nv_bfloat16>(p, K, V, stream) : bwd::launch_io<float>(p, K, V, stream);
}

}  // namespace kda
