// kda_recurrent.cu -- token-recurrent KDA forward on CUDA cores, fp32 state.
//
// Evaluates the defining recurrence directly (page "手撕KDA", section "1 Naive":
// the recurrence that naive_chunk_kda evaluates chunk-wise):
//     P   = Diag(exp g_t) S_{t-1}
//     u   = P^T k_t
//     S_t = P + beta_t k_t (v_t - u)^T          ( = (I - b k k^T) P + b k v^T )
//     o_t = scale S_t^T q_t
// One block per (value-column slice of 32, value head, sequence): the K x 32
// slice of S lives in registers (8 warps x K/8 rows, lane = column), the two
// reductions over K per token go through shared memory, and the next token's
// inputs are staged while the current one is processed (two barriers/token).
// Used for fp32 I/O (where bf16 tensor-core operands cannot meet fp32
// accuracy) and for shapes the tensor-core kernel does not cover.
#include "kda_common.cuh"

namespace kda {

template <typename IO, int K>
__global__ void __launch_bounds__(256) recurrent_fwd_kernel(FwdParams p) {
  constexpr int NW = 8;
  constexpr int RPW = K / NW;  // state rows per warp
  const int slice = blockIdx.x, hv = blockIdx.y, seq = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int V = p.V, HV = p.HV, H = p.H;
  const int hk = hv / (HV / H);
  const int col = slice * 32 + lane;

  __shared__ float s_k[2][K], s_q[2][K], s_g[2][K], s_v[2][32], s_b[2];
  __shared__ float red_u[NW][32];
  __shared__ float red_o[2][NW][32];

  long tok0;
  int len;
  seq_range(p, seq, tok0, len);

  float s[RPW];
  const size_t state_off = (static_cast<size_t>(seq) * HV + hv) * K * V;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int d = warp * RPW + r;
    s[r] = p.s0 ? p.s0[state_off + static_cast<size_t>(d) * V + col] : 0.f;
  }

  const IO* q = static_cast<const IO*>(p.q);
  const IO* k = static_cast<const IO*>(p.k);
  const IO* v = static_cast<const IO*>(p.v);
  IO* out = static_cast<IO*>(p.out);

  auto stage = [&](int t, int buf) {
    const size_t tok = static_cast<size_t>(tok0 + t);
    const int i = threadIdx.x;
    if (i < K) {
      s_k[buf][i] = to_f32(k[(tok * H + hk) * K + i]);
      s_q[buf][i] = to_f32(q[(tok * H + hk) * K + i]);
      s_g[buf][i] = p.g[(tok * HV + hv) * K + i];
    } else if (i < K + 32) {
      s_v[buf][i - K] = to_f32(v[(tok * HV + hv) * V + slice * 32 + (i - K)]);
    } else if (i == K + 32) {
      s_b[buf] = p.beta[tok * HV + hv];
    }
  };
  auto emit = [&](int t) {  // warp 0: finish the reduction for o_t and store it
    const int b = t & 1;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) acc += red_o[b][w][lane];
    const size_t tok = static_cast<size_t>(tok0 + t);
    out[(tok * HV + hv) * V + col] = from_f32<IO>(p.scale * acc);
  };

  if (len > 0) stage(0, 0);
  __syncthreads();
  for (int t = 0; t < len; ++t) {
    const int buf = t & 1;
    // phase A: decay the state rows, partial u = P^T k, stage the next token
    float pu = 0.f;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int d = warp * RPW + r;
      s[r] *= expf(s_g[buf][d]);
      pu = fmaf(s_k[buf][d], s[r], pu);
    }
    red_u[warp][lane] = pu;
    if (t + 1 < len) stage(t + 1, buf ^ 1);
    if (warp == 0 && t > 0) emit(t - 1);
    __syncthreads();
    // phase B: u, rank-1 correction, partial o = S^T q
    float u = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) u += red_u[w][lane];
    const float bv = s_b[buf] * (s_v[buf][lane] - u);
    float po = 0.f;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int d = warp * RPW + r;
      s[r] = fmaf(s_k[buf][d], bv, s[r]);
      po = fmaf(s_q[buf][d], s[r], po);
    }
    red_o[buf][warp][lane] = po;
    __syncthreads();
  }
  if (warp == 0 && len > 0) emit(len - 1);

  if (p.sfin) {
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      const int d = warp * RPW + r;
      p.sfin[state_off + static_cast<size_t>(d) * V + col] = s[r];
    }
  }
}

// Host launcher (called from the ABI layer after validation).
cudaError_t launch_recurrent_fwd(const FwdParams& p, bool bf16, cudaStream_t stream) {
  const int ns = p.cu ? p.num_seqs : p.num_seqs;  // caller sets num_seqs = B when not varlen
  dim3 grid(p.V / 32, p.HV, ns);
  if (bf16) {
    if (p.K == 128) recurrent_fwd_kernel<__nv_bfloat16, 128><<<grid, 256, 0, stream>>>(p);
    else recurrent_fwd_kernel<__nv_bfloat16, 64><<<grid, 256, 0, stream>>>(p);
  } else {
    if (p.K == 128) recurrent_fwd_kernel<float, 128><<<grid, 256, 0, stream>>>(p);
    else recurrent_fwd_kernel<float, 64><<<grid, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kda
