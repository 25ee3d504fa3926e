// kda_decode.cu -- the recurrent step for inference: a few tokens per sequence
// against a resident fp32 state, updated in place.
//
// For each (sequence, value head) and each of the call's T tokens (page "手撕KDA",
// section "1 Naive": the recurrence that naive_chunk_kda evaluates chunk-wise;
// section 5 validates the chunked kernels against this recurrent form):
//     P   = Diag(exp g_t) S
//     u   = P^T k_t
//     S   = P + beta_t k_t (v_t - u)^T          ( = (I - beta k k^T) P + beta k v^T )
//     o_t = scale S^T q_t
// At T = 1 the step reads and writes the K x V state once (128 KiB per (sequence,
// value head) at K = V = 128) and a few hundred bytes of inputs: it is bound by HBM
// bandwidth on the state, so the kernel is built around moving the state at full
// width: one CTA per (sequence, value head), 256 threads, each holding 4 adjacent
// value columns of K / (1024 / V) state rows in registers, every state row read and
// written as 16-byte vectors by consecutive threads.  The two reductions over K per
// token go through shared memory (double-buffered, two barriers per token).
#include "kda_common.cuh"

namespace kda {
namespace dec {

constexpr int NT = 256;

struct Params {
  const void* q;     // [B, T, H, K]  io type
  const void* k;     // [B, T, H, K]
  const void* v;     // [B, T, HV, V]
  const float* g;    // [B, T, HV, K]
  const float* beta; // [B, T, HV]
  float* state;      // [B, HV, K, V] fp32, read and written in place
  void* out;         // [B, T, HV, V] io type
  float scale;
  int T, H, HV;
};

template <typename IO, int K, int V>
__global__ void __launch_bounds__(NT) decode_kernel(const Params p) {
  constexpr int TPR = V / 4;        // threads across one state row (4 columns each)
  constexpr int RG = NT / TPR;      // row groups
  constexpr int RPT = K / RG;       // state rows per thread
  static_assert(RPT * RG == K && TPR * 4 == V, "decode tiling");
  const int hv = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x;
  const int cg = tid % TPR;         // column group: columns 4 cg .. 4 cg + 3
  const int rg = tid / TPR;         // row group: rows rg, rg + RG, ... (interleaved)
  const int hk = hv / (p.HV / p.H);

  __shared__ float s_k[2][K], s_q[2][K], s_e[2][K], s_v[2][V], s_b[2];
  __shared__ __align__(16) float red_u[RG][V];
  __shared__ __align__(16) float red_o[2][RG][V];

  const IO* q = static_cast<const IO*>(p.q);
  const IO* k = static_cast<const IO*>(p.k);
  const IO* v = static_cast<const IO*>(p.v);
  IO* out = static_cast<IO*>(p.out);
  float* st = p.state + (static_cast<size_t>(b) * p.HV + hv) * K * V + 4 * cg;

  // the state slice in registers: rows rg + RG i, columns 4 cg .. 4 cg + 3
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = *reinterpret_cast<const float4*>(st + static_cast<size_t>(rg + RG * i) * V);

  auto stage = [&](int t, int buf) {
    const size_t tok = static_cast<size_t>(b) * p.T + t;
    if (tid < K) {
      s_k[buf][tid] = to_f32(k[(tok * p.H + hk) * K + tid]);
      s_q[buf][tid] = to_f32(q[(tok * p.H + hk) * K + tid]);
      s_e[buf][tid] = expf(p.g[(tok * p.HV + hv) * K + tid]);
    } else if (tid < K + V) {
      s_v[buf][tid - K] = to_f32(v[(tok * p.HV + hv) * V + (tid - K)]);
    }
    if (tid == NT - 1) s_b[buf] = p.beta[tok * p.HV + hv];
  };
  auto emit = [&](int t) {  // row group 0: finish o_t for its 4 columns and store them
    const int buf = t & 1;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(&red_o[buf][r][4 * cg]);
      acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
    }
    const size_t o_off = ((static_cast<size_t>(b) * p.T + t) * p.HV + hv) * V + 4 * cg;
#pragma unroll
    for (int c = 0; c < 4; ++c) out[o_off + c] = from_f32<IO>(p.scale * (&acc.x)[c]);
  };

  if (p.T > 0) stage(0, 0);
  __syncthreads();
  for (int t = 0; t < p.T; ++t) {
    const int buf = t & 1;
    // decay the rows, partial u = P^T k over this thread's rows; stage the next token
    float4 pu = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int d = rg + RG * i;
      const float e = s_e[buf][d], kd = s_k[buf][d];
      s[i].x *= e; s[i].y *= e; s[i].z *= e; s[i].w *= e;
      pu.x = fmaf(kd, s[i].x, pu.x); pu.y = fmaf(kd, s[i].y, pu.y);
      pu.z = fmaf(kd, s[i].z, pu.z); pu.w = fmaf(kd, s[i].w, pu.w);
    }
    *reinterpret_cast<float4*>(&red_u[rg][4 * cg]) = pu;
    if (t + 1 < p.T) stage(t + 1, buf ^ 1);
    if (rg == 0 && t > 0) emit(t - 1);
    __syncthreads();
    // u, the rank-1 correction, partial o = S^T q
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(&red_u[r][4 * cg]);
      u.x += x.x; u.y += x.y; u.z += x.z; u.w += x.w;
    }
    const float bt = s_b[buf];
    const float4 bv = make_float4(bt * (s_v[buf][4 * cg] - u.x), bt * (s_v[buf][4 * cg + 1] - u.y),
                                  bt * (s_v[buf][4 * cg + 2] - u.z), bt * (s_v[buf][4 * cg + 3] - u.w));
    float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int d = rg + RG * i;
      const float kd = s_k[buf][d], qd = s_q[buf][d];
      s[i].x = fmaf(kd, bv.x, s[i].x); s[i].y = fmaf(kd, bv.y, s[i].y);
      s[i].z = fmaf(kd, bv.z, s[i].z); s[i].w = fmaf(kd, bv.w, s[i].w);
      po.x = fmaf(qd, s[i].x, po.x); po.y = fmaf(qd, s[i].y, po.y);
      po.z = fmaf(qd, s[i].z, po.z); po.w = fmaf(qd, s[i].w, po.w);
    }
    *reinterpret_cast<float4*>(&red_o[buf][rg][4 * cg]) = po;
    __syncthreads();
  }
  if (rg == 0 && p.T > 0) emit(p.T - 1);
#pragma unroll
  for (int i = 0; i < RPT; ++i) *reinterpret_cast<float4*>(st + static_cast<size_t>(rg + RG * i) * V) = s[i];
}

template <typename IO>
cudaError_t launch_io(const Params& p, int K, int V, int B, cudaStream_t stream) {
  const dim3 grid(p.HV, B);
  if (K == 128 && V == 128) decode_kernel<IO, 128, 128><<<grid, NT, 0, stream>>>(p);
  else if (K == 128 && V == 64) decode_kernel<IO, 128, 64><<<grid, NT, 0, stream>>>(p);
  else if (K == 64 && V == 128) decode_kernel<IO, 64, 128><<<grid, NT, 0, stream>>>(p);
  else decode_kernel<IO, 64, 64><<<grid, NT, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dec

// Host launcher (called from the ABI layer after validation).
cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          float* state, void* out, float scale, int B, int T, int H, int HV, int K, int V,
                          bool bf16, cudaStream_t stream) {
  dec::Params p{q, k, v, g, beta, state, out, scale, T, H, HV};
  return bf16 ? dec::launch_io<__nv_bfloat16>(p, K, V, B, stream) : dec::launch_io<float>(p, K, V, B, stream);
}

}  // namespace kda
