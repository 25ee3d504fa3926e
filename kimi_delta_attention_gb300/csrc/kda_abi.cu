// kda_abi.cu -- the C ABI declared in include/kda.h: host-side validation,
// workspace sizing, status reporting and dispatch to the forward kernels.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/kda.h"
#include "kda_common.cuh"

namespace kda {
cudaError_t launch_recurrent_fwd(const FwdParams& p, bool bf16, cudaStream_t stream);
bool chunk_tc_supported(const FwdParams& p, bool bf16);
size_t chunk_tc_ring_bytes(int num_seqs, int HV);
cudaError_t launch_chunk_tc_fwd(const FwdParams& p, cudaStream_t stream);
const char* chunk_kernel_name(bool bf16, int K, int V, long tokens, int num_seqs, int HV, bool packed);
int chunk_kernel_launches(bool bf16, int K, int V, long tokens, int num_seqs, int HV, bool packed);
cudaError_t launch_chunk_output(const FwdParams& p, cudaStream_t stream);
size_t backward_unit_floats(long max_len, int K, int V);
cudaError_t launch_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const float* s0, const int32_t* cu, const void* d_out, const float* d_fin, float* dq,
                            float* dk, float* dv, float* dg, float* dbeta, float* ds0, float* scratch,
                            size_t unit_floats, uint32_t* status, float scale, int T, int H, int HV, int K, int V,
                            int num_seqs, bool bf16, cudaStream_t stream);
size_t backward_chunk_slots(long T, int num_seqs_or_B, bool varlen, int HV);
size_t backward_chunk_slot_floats(int K, int V);
cudaError_t launch_backward_chunk(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  const float* s0, const int32_t* cu, const void* d_out, const float* d_fin, float* dq,
                                  float* dk, float* dv, float* dg, float* dbeta, float* ds0, float* ws,
                                  uint32_t* status, unsigned long long wait_ns, float scale, int T, int H, int HV,
                                  int K, int V, int num_seqs, bool bf16, cudaStream_t stream);
cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          float* state, void* out, float scale, int B, int T, int H, int HV, int K, int V,
                          bool bf16, cudaStream_t stream);
}  // namespace kda

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Workspace bytes an entry point needs: the status word, plus the record ring
// when the tensor-core chunk kernel will run.
size_t workspace_needed(const kda_shape* s, bool use_tc) {
  if (!s) return kda::kWorkspaceBytes;
  const bool tc = use_tc && s->io_dtype == KDA_BF16 && s->K == 128 && s->V == 128 && s->HV >= 1;
  if (!tc) return kda::kWorkspaceBytes;
  const int ns = s->num_seqs > 0 ? s->num_seqs : s->B;
  if (ns <= 0) return kda::kWorkspaceBytes;
  return kda::kRingOffset + kda::chunk_tc_ring_bytes(ns, s->HV);
}

// Limit of the kernels' bounded waits for work: 2 s, or KDA_WAIT_LIMIT_NS (a positive
// integer, read at each call) for tests that make those waits run out.
unsigned long long wait_limit_ns() {
  const char* e = std::getenv("KDA_WAIT_LIMIT_NS");
  if (e) {
    char* end = nullptr;
    const unsigned long long v = std::strtoull(e, &end, 10);
    if (end != e && v > 0) return v;
  }
  return 2000000000ull;
}

// KDA_BACKWARD=recurrent (read at each call) selects the token-recurrence backward.
bool backward_recurrent() {
  const char* e = std::getenv("KDA_BACKWARD");
  return e && std::strcmp(e, "recurrent") == 0;
}

struct Checked {
  kda::FwdParams p;
  bool bf16;
  size_t units;  // sequences * value heads
};

// g_elem: bytes per element of g (4: the log-space decay; 2: the gated entry's bf16 gate input)
kda_status validate(bool use_tc, const kda_shape* s, const void* q, const void* k, const void* v,
                    const void* g, const float* beta, float scale, const float* s0, const int32_t* cu,
                    void* out, float* sfin, void* ws, size_t ws_bytes, Checked& c, size_t g_elem = 4) {
  if (!s) return KDA_ERR_INVALID_ARG;
  if (s->B < 0 || s->T < 0 || s->H < 1 || s->HV < 1 || s->K < 1 || s->V < 1) return KDA_ERR_INVALID_ARG;
  if (s->HV % s->H != 0) return KDA_ERR_INVALID_ARG;
  if (s->io_dtype != KDA_F32 && s->io_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
  if (cu) {
    if (s->B != 1 || s->num_seqs < 1) return KDA_ERR_INVALID_ARG;
  } else if (s->num_seqs != 0) {
    return KDA_ERR_INVALID_ARG;
  }
  if ((s->K != 64 && s->K != 128) || (s->V != 64 && s->V != 128)) return KDA_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < workspace_needed(s, use_tc)) return KDA_ERR_WORKSPACE;

  const size_t ns = cu ? static_cast<size_t>(s->num_seqs) : static_cast<size_t>(s->B);
  const size_t tokens = cu ? static_cast<size_t>(s->T) : static_cast<size_t>(s->B) * s->T;
  const size_t es = s->io_dtype == KDA_BF16 ? 2 : 4;
  const size_t n_qk = tokens * s->H * s->K * es, n_v = tokens * s->HV * s->V * es;
  const size_t n_g = tokens * s->HV * s->K * g_elem, n_b = tokens * s->HV * 4;
  const size_t n_s = ns * s->HV * s->K * s->V * 4;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
  // tensors read or written in 16-byte vectors / TMA tiles need 16-byte
  // alignment; beta and cu_seqlens are read one element at a time
  const void* ptrs16[] = {q, k, v, g, s0, out, sfin, ws};
  for (const void* ptr : ptrs16)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  if ((beta && !aligned(beta, 4)) || (cu && !aligned(cu, 4))) return KDA_ERR_ALIGNMENT;
  // out must not alias an input; final_state may alias initial_state only exactly
  const void* ins[] = {q, k, v, g, beta, s0};
  const size_t nins[] = {n_qk, n_qk, n_v, n_g, n_b, n_s};
  for (int i = 0; i < 6; ++i) {
    if (overlaps(out, n_v, ins[i], nins[i])) return KDA_ERR_INVALID_ARG;
    if (i < 5 && overlaps(sfin, n_s, ins[i], nins[i])) return KDA_ERR_INVALID_ARG;
  }
  if (sfin && s0 && sfin != s0 && overlaps(sfin, n_s, s0, n_s)) return KDA_ERR_INVALID_ARG;
  if (overlaps(sfin, n_s, out, n_v) || overlaps(ws, ws_bytes, out, n_v) || overlaps(ws, ws_bytes, sfin, n_s))
    return KDA_ERR_INVALID_ARG;

  kda::FwdParams& p = c.p;
  std::memset(&p, 0, sizeof(p));
  p.q = q; p.k = k; p.v = v; p.g = static_cast<const float*>(g); p.beta = beta; p.s0 = s0; p.cu = cu;
  p.out = out; p.sfin = sfin; p.status = static_cast<uint32_t*>(ws);
  p.ring = ws_bytes > kda::kRingOffset ? static_cast<uint8_t*>(ws) + kda::kRingOffset : nullptr;
  p.wait_ns = wait_limit_ns();
  p.scale = scale; p.T = s->T; p.H = s->H; p.HV = s->HV; p.K = s->K; p.V = s->V;
  p.num_seqs = static_cast<int>(ns);
  c.bf16 = s->io_dtype == KDA_BF16;
  c.units = ns * s->HV;
  return KDA_OK;
}

kda_status run(bool use_tc, const kda_shape* s, const void* q, const void* k, const void* v,
               const float* g, const float* beta, float scale, const float* s0, const int32_t* cu,
               void* out, float* sfin, void* ws, size_t ws_bytes, void* stream) {
  Checked c;
  const kda_status st = validate(use_tc, s, q, k, v, g, beta, scale, s0, cu, out, sfin, ws, ws_bytes, c);
  if (st != KDA_OK) return st;
  if (c.units == 0) return KDA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (use_tc && c.p.ring && kda::chunk_tc_supported(c.p, c.bf16)) {
    e = kda::launch_chunk_tc_fwd(c.p, cs);  // resets the status word itself
  } else {
    if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), cs) != cudaSuccess) return KDA_ERR_CUDA;
    e = kda::launch_recurrent_fwd(c.p, c.bf16, cs);
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// ---- fixed scratch for kda_chunk_fwd_static_scratch ----
constexpr size_t kStaticScratchBytes =
    kda::kRingOffset + static_cast<size_t>(KDA_STATIC_SCRATCH_MAX_UNITS) * kda::kRingBytesPerUnit;

// One copy per device that loads the library, alive until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
uint8_t* g_static_ptr[kMaxDevices] = {};

// Device address of the current device's array; looked up once per device
// with that device current (host code may not use the symbol itself).
uint8_t* static_scratch_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return nullptr;
    g_static_ptr[dev] = static_cast<uint8_t*>(ptr);
  }
  return g_static_ptr[dev];
}

}  // namespace

extern "C" {

kda_status kda_chunk_fwd(const kda_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, float scale, const float* initial_state,
                         const int32_t* cu_seqlens, void* out, float* final_state, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return run(true, shape, q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, workspace,
             workspace_bytes, stream);
}

kda_status kda_recurrent_fwd(const kda_shape* shape, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, float scale, const float* initial_state,
                             const int32_t* cu_seqlens, void* out, float* final_state, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return run(false, shape, q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, workspace,
             workspace_bytes, stream);
}

size_t kda_chunk_fwd_workspace_size(const kda_shape* shape) { return workspace_needed(shape, true); }

kda_status kda_read_device_status(const void* workspace, void* stream) {
  if (!workspace) return KDA_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return KDA_ERR_CUDA;
  if (word & kda::kStatusTimeout) return KDA_ERR_DEVICE_TIMEOUT;
  if (word & kda::kStatusBounds) return KDA_ERR_DEVICE_BOUNDS;
  if (word & kda::kStatusRange) return KDA_ERR_DECAY_RANGE;
  return KDA_OK;
}

const char* kda_status_string(kda_status status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape (K and V must be 64 or 128)";
    case KDA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case KDA_ERR_CUDA: return "CUDA runtime error";
    case KDA_ERR_DEVICE_TIMEOUT: return "device: a bounded on-chip wait timed out";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_DEVICE_BOUNDS: return "device: cu_seqlens out of order or out of range";
    case KDA_ERR_STATIC_SCRATCH: return "more (sequence, value head) pairs than the static scratch holds";
    case KDA_ERR_DECAY_RANGE: return "device: g decays faster than the chunk kernels support (16-token sum < -83)";
  }
  return "unknown status";
}

int kda_chunk_size(void) { return 64; }

const char* kda_chunk_fwd_kernel_name(const kda_shape* s) {
  if (!s || s->B < 0 || s->T < 0 || s->HV < 1 || s->num_seqs < 0) return "none";
  const long ns = s->num_seqs > 0 ? s->num_seqs : s->B;
  const long tokens = s->num_seqs > 0 ? static_cast<long>(s->T) : static_cast<long>(s->B) * s->T;
  if (ns * s->HV > (1L << 30) || ns == 0) return "none";
  return kda::chunk_kernel_name(s->io_dtype == KDA_BF16, s->K, s->V, tokens, static_cast<int>(ns), s->HV,
                                s->num_seqs > 0);
}

int kda_chunk_fwd_kernel_launches(const kda_shape* s) {
  if (!s || s->B < 0 || s->T < 0 || s->HV < 1 || s->num_seqs < 0) return 0;
  const long ns = s->num_seqs > 0 ? s->num_seqs : s->B;
  const long tokens = s->num_seqs > 0 ? static_cast<long>(s->T) : static_cast<long>(s->B) * s->T;
  if (ns * s->HV > (1L << 30) || ns == 0) return 0;
  return kda::chunk_kernel_launches(s->io_dtype == KDA_BF16, s->K, s->V, tokens, static_cast<int>(ns), s->HV,
                                    s->num_seqs > 0);
}

kda_status kda_chunk_fwd_gated(const kda_shape* shape, const void* q, const void* k, const void* v,
                               const void* g_raw, const float* beta_raw, const kda_gate* gate, float scale,
                               const float* initial_state, const int32_t* cu_seqlens, void* out,
                               float* final_state, void* workspace, size_t workspace_bytes, void* stream) {
  if (!shape || !gate) return KDA_ERR_INVALID_ARG;
  if (gate->kind != KDA_GATE_BOUNDED && gate->kind != KDA_GATE_SOFTPLUS) return KDA_ERR_INVALID_ARG;
  if (gate->kind == KDA_GATE_BOUNDED && !(gate->lower_bound < 0.f && std::isfinite(gate->lower_bound)))
    return KDA_ERR_INVALID_ARG;
  if (!gate->A_log || !gate->dt_bias) return KDA_ERR_INVALID_ARG;
  if (!aligned(gate->A_log, 4) || !aligned(gate->dt_bias, 16)) return KDA_ERR_ALIGNMENT;
  // g_raw (bf16) takes the place of g in the common checks, at its own size
  Checked c;
  kda_status st = validate(true, shape, q, k, v, g_raw, beta_raw, scale, initial_state, cu_seqlens, out,
                           final_state, workspace, workspace_bytes, c, 2);
  if (st != KDA_OK) return st;
  if (c.units == 0) return KDA_OK;
  const long tokens = cu_seqlens ? static_cast<long>(shape->T) : static_cast<long>(shape->B) * shape->T;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (tokens == 0) {  // nothing to activate: the state copy of an empty forward
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), cs) != cudaSuccess) return KDA_ERR_CUDA;
    return kda::launch_recurrent_fwd(c.p, c.bf16, cs) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  if (!c.p.ring || !kda::chunk_tc_supported(c.p, c.bf16)) return KDA_ERR_UNSUPPORTED;
  c.p.prestage = gate->kind == KDA_GATE_BOUNDED ? 1 : 2;
  c.p.g_raw = static_cast<const uint16_t*>(g_raw);
  c.p.g = nullptr;
  c.p.A_log = gate->A_log;
  c.p.dt_bias = gate->dt_bias;
  c.p.lower_bound = gate->lower_bound;
  return kda::launch_chunk_tc_fwd(c.p, cs) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_chunk_states_size(const kda_shape* s) {
  if (!s || s->B < 0 || s->T < 0 || s->HV < 1 || s->K < 1 || s->V < 1 || s->num_seqs != 0) return 0;
  const size_t nt = (static_cast<size_t>(s->T) + 63) / 64;
  return static_cast<size_t>(s->B) * s->HV * nt * s->K * s->V * 2;
}

namespace {
// The state pass and the output kernel take fixed-length bf16 batches at K = V = 128.
kda_status states_shape_ok(const kda_shape* s) {
  if (!s) return KDA_ERR_INVALID_ARG;
  if (s->num_seqs != 0) return KDA_ERR_UNSUPPORTED;
  if (s->io_dtype != KDA_BF16 || s->K != 128 || s->V != 128) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}
}  // namespace

kda_status kda_chunk_states(const kda_shape* shape, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* initial_state, void* h, float* final_state,
                            void* workspace, size_t workspace_bytes, void* stream) {
  kda_status st = states_shape_ok(shape);
  if (st != KDA_OK) return st;
  if (!h && shape->B > 0 && shape->T > 0) return KDA_ERR_INVALID_ARG;
  // h takes the place of the output in the common checks (alignment, overlaps at o's size),
  // then is checked at its own size
  Checked c;
  st = validate(true, shape, q, k, v, g, beta, 1.f, initial_state, nullptr, h, final_state, workspace,
                workspace_bytes, c);
  if (st != KDA_OK) return st;
  const size_t nh = kda_chunk_states_size(shape);
  const size_t tokens = static_cast<size_t>(shape->B) * shape->T;
  const size_t n_qk = tokens * shape->H * shape->K * 2, n_v = tokens * shape->HV * shape->V * 2;
  const size_t n_g = tokens * shape->HV * shape->K * 4, n_b = tokens * shape->HV * 4;
  const size_t n_s = static_cast<size_t>(shape->B) * shape->HV * shape->K * shape->V * 4;
  const void* others[] = {q, k, v, g, beta, initial_state, final_state, workspace};
  const size_t nothers[] = {n_qk, n_qk, n_v, n_g, n_b, n_s, n_s, workspace_bytes};
  for (int i = 0; i < 8; ++i)
    if (overlaps(h, nh, others[i], nothers[i])) return KDA_ERR_INVALID_ARG;
  if (c.units == 0) return KDA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (tokens == 0) {  // no chunks: the final state is the initial one
    c.p.out = nullptr;
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), cs) != cudaSuccess) return KDA_ERR_CUDA;
    return kda::launch_recurrent_fwd(c.p, true, cs) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  if (!c.p.ring || !kda::chunk_tc_supported(c.p, c.bf16)) return KDA_ERR_UNSUPPORTED;
  c.p.out = nullptr;
  c.p.h = static_cast<uint16_t*>(h);
  c.p.h_chunks = static_cast<int>((shape->T + 63) / 64);
  return kda::launch_chunk_tc_fwd(c.p, cs) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_chunk_output(const kda_shape* shape, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float scale, const void* h, void* out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  kda_status st = states_shape_ok(shape);
  if (st != KDA_OK) return st;
  Checked c;
  st = validate(false, shape, q, k, v, g, beta, scale, nullptr, nullptr, out, nullptr, workspace, workspace_bytes, c);
  if (st != KDA_OK) return st;
  const size_t tokens = static_cast<size_t>(shape->B) * shape->T;
  if (c.units == 0 || tokens == 0) return KDA_OK;
  if (!h) return KDA_ERR_INVALID_ARG;
  if (!aligned(h, 16)) return KDA_ERR_ALIGNMENT;
  const size_t nh = kda_chunk_states_size(shape);
  if (overlaps(h, nh, out, tokens * shape->HV * shape->V * 2) || overlaps(h, nh, workspace, workspace_bytes))
    return KDA_ERR_INVALID_ARG;
  if (!kda::chunk_tc_supported(c.p, c.bf16)) return KDA_ERR_UNSUPPORTED;
  c.p.h = static_cast<uint16_t*>(const_cast<void*>(h));
  c.p.h_chunks = static_cast<int>((shape->T + 63) / 64);
  return kda::launch_chunk_output(c.p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_backward_workspace_size(const kda_shape* s) {
  if (!s || s->B < 0 || s->T < 0 || s->HV < 1 || s->K < 1 || s->V < 1 || s->num_seqs < 0) return 0;
  const size_t ns = s->num_seqs > 0 ? s->num_seqs : s->B;
  const size_t recurrent = ns * s->HV * kda::backward_unit_floats(s->T, s->K, s->V);
  const size_t chunk = kda::backward_chunk_slots(s->T, static_cast<int>(ns), s->num_seqs > 0, s->HV) *
                       kda::backward_chunk_slot_floats(s->K, s->V);
  return 256 + (recurrent > chunk ? recurrent : chunk) * sizeof(float);
}

kda_status kda_backward(const kda_shape* s, const void* q, const void* k, const void* v, const float* g,
                        const float* beta, float scale, const float* initial_state, const int32_t* cu_seqlens,
                        const void* d_out, const float* d_final_state, float* dq, float* dk, float* dv, float* dg,
                        float* dbeta, float* d_initial_state, void* workspace, size_t workspace_bytes,
                        void* stream) {
  // the forward's own checks (shapes, alignment, aliasing among the inputs) with d_out in the
  // place of the output; the gradients are then checked against everything else
  Checked c;
  kda_status st = validate(false, s, q, k, v, g, beta, scale, initial_state, cu_seqlens, const_cast<void*>(d_out),
                           nullptr, workspace, workspace_bytes, c);
  if (st != KDA_OK) return st;
  if (workspace_bytes < kda_backward_workspace_size(s)) return KDA_ERR_WORKSPACE;
  const size_t ns = cu_seqlens ? static_cast<size_t>(s->num_seqs) : static_cast<size_t>(s->B);
  const size_t tokens = cu_seqlens ? static_cast<size_t>(s->T) : static_cast<size_t>(s->B) * s->T;
  const size_t es = s->io_dtype == KDA_BF16 ? 2 : 4;
  const size_t n_qk = tokens * s->H * s->K * es, n_v = tokens * s->HV * s->V * es;
  const size_t n_g = tokens * s->HV * s->K * 4, n_b = tokens * s->HV * 4, n_s = ns * s->HV * s->K * s->V * 4;
  const size_t f_qk = tokens * s->H * s->K * 4, f_v = tokens * s->HV * s->V * 4;
  if (tokens > 0 && (!dq || !dk || !dv || !dg || !dbeta)) return KDA_ERR_INVALID_ARG;
  const void* outs[] = {dq, dk, dv, dg, dbeta, d_initial_state};
  const size_t nouts[] = {f_qk, f_qk, f_v, n_g, n_b, n_s};
  for (const void* ptr : outs)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  if (d_final_state && !aligned(d_final_state, 16)) return KDA_ERR_ALIGNMENT;
  const void* ins[] = {q, k, v, g, beta, initial_state, d_out, d_final_state, workspace};
  const size_t nins[] = {n_qk, n_qk, n_v, n_g, n_b, n_s, n_v, n_s, workspace_bytes};
  for (int j = 0; j < 8; ++j)  // the scratch is written while the inputs are read
    if (overlaps(workspace, workspace_bytes, ins[j], nins[j])) return KDA_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i) {
    for (int j = 0; j < 9; ++j)
      if (overlaps(outs[i], nouts[i], ins[j], nins[j])) return KDA_ERR_INVALID_ARG;
    for (int j = i + 1; j < 6; ++j)
      if (overlaps(outs[i], nouts[i], outs[j], nouts[j])) return KDA_ERR_INVALID_ARG;
  }
  if (c.units == 0) return KDA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint32_t* status = static_cast<uint32_t*>(workspace);
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), cs) != cudaSuccess) return KDA_ERR_CUDA;
  // dq and dk gather the value heads that share a key head, and dq, dk, dg and dbeta the
  // kernel's value-column slices: zero them first
  if (tokens > 0 && (cudaMemsetAsync(dq, 0, f_qk, cs) != cudaSuccess || cudaMemsetAsync(dk, 0, f_qk, cs) != cudaSuccess ||
                     cudaMemsetAsync(dg, 0, n_g, cs) != cudaSuccess || cudaMemsetAsync(dbeta, 0, n_b, cs) != cudaSuccess))
    return KDA_ERR_CUDA;
  float* scratch = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256);
  if (!backward_recurrent()) {
    const cudaError_t e = kda::launch_backward_chunk(
        q, k, v, g, beta, initial_state, cu_seqlens, d_out, d_final_state, dq, dk, dv, dg, dbeta, d_initial_state,
        scratch, status, wait_limit_ns(), scale, s->T, s->H, s->HV, s->K, s->V, static_cast<int>(ns),
        s->io_dtype == KDA_BF16, cs);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  }
  const cudaError_t e = kda::launch_backward(
      q, k, v, g, beta, initial_state, cu_seqlens, d_out, d_final_state, dq, dk, dv, dg, dbeta, d_initial_state,
      scratch, kda::backward_unit_floats(s->T, s->K, s->V), status, scale, s->T, s->H, s->HV, s->K, s->V,
      static_cast<int>(ns), s->io_dtype == KDA_BF16, cs);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_decode(const kda_shape* s, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, float* state, void* out, void* stream) {
  if (!s) return KDA_ERR_INVALID_ARG;
  if (s->B < 0 || s->T < 0 || s->H < 1 || s->HV < 1 || s->K < 1 || s->V < 1 || s->num_seqs != 0)
    return KDA_ERR_INVALID_ARG;
  if (s->HV % s->H != 0) return KDA_ERR_INVALID_ARG;
  if (s->io_dtype != KDA_F32 && s->io_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
  if ((s->K != 64 && s->K != 128) || (s->V != 64 && s->V != 128)) return KDA_ERR_UNSUPPORTED;
  const size_t B = static_cast<size_t>(s->B), tokens = B * s->T;
  const size_t es = s->io_dtype == KDA_BF16 ? 2 : 4;
  const size_t n_qk = tokens * s->H * s->K * es, n_v = tokens * s->HV * s->V * es;
  const size_t n_g = tokens * s->HV * s->K * 4, n_b = tokens * s->HV * 4;
  const size_t n_s = B * s->HV * s->K * s->V * 4;
  if (B == 0) return KDA_OK;
  if (!state) return KDA_ERR_INVALID_ARG;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
  const void* ptrs16[] = {q, k, v, g, out, state};
  for (const void* ptr : ptrs16)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  if (beta && !aligned(beta, 4)) return KDA_ERR_ALIGNMENT;
  const void* ins[] = {q, k, v, g, beta};
  const size_t nins[] = {n_qk, n_qk, n_v, n_g, n_b};
  for (int i = 0; i < 5; ++i)
    if (overlaps(out, n_v, ins[i], nins[i]) || overlaps(state, n_s, ins[i], nins[i])) return KDA_ERR_INVALID_ARG;
  if (overlaps(state, n_s, out, n_v)) return KDA_ERR_INVALID_ARG;
  const cudaError_t e = kda::launch_decode(q, k, v, g, beta, state, out, scale, s->B, s->T, s->H, s->HV, s->K,
                                           s->V, s->io_dtype == KDA_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_chunk_fwd_static_scratch(const kda_shape* shape, const void* q, const void* k, const void* v,
                                        const float* g, const float* beta, float scale,
                                        const float* initial_state, const int32_t* cu_seqlens, void* out,
                                        float* final_state, void* stream, void** status_word) {
  if (!shape) return KDA_ERR_INVALID_ARG;
  const long ns = shape->num_seqs > 0 ? shape->num_seqs : shape->B;
  if (ns < 0 || shape->HV < 1) return KDA_ERR_INVALID_ARG;
  if (ns * static_cast<long>(shape->HV) > KDA_STATIC_SCRATCH_MAX_UNITS) return KDA_ERR_STATIC_SCRATCH;
  uint8_t* scratch = static_scratch_current_device();
  if (!scratch) return KDA_ERR_CUDA;
  if (status_word) *status_word = scratch;
  return run(true, shape, q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, scratch,
             kStaticScratchBytes, stream);
}

}  // extern "C"
