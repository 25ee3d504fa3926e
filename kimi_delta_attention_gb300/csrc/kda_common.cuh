// kda_common.cuh -- launch parameters and small helpers shared by the KDA
// forward kernels (CUDA library side only).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace kda {

// Device status word bits (the first 32-bit word of the workspace).
constexpr uint32_t kStatusTimeout = 1u;   // a bounded on-chip wait gave up
constexpr uint32_t kStatusBounds = 2u;    // cu_seqlens entry out of order / range
constexpr uint32_t kStatusRange = 4u;     // a 16-token block of g decays faster than the chunk kernels support

// Workspace layout: [0, 4) status word, [8, kFlagOffset) optional profile counters,
// [kFlagOffset, kFlagOffset + kMaxSplitUnits * kFlagBytesPerUnit) the record
// flags of the split chunk kernel (zeroed before each launch that uses them);
// the tensor-core chunk kernels' record rings start at kRingOffset.
constexpr size_t kWorkspaceBytes = 256;   // minimum (status word only)
constexpr size_t kFlagOffset = 4096;
static_assert(kFlagOffset >= 512 * 8, "profile words (uint64 [1, 512)) stay below the flags");
constexpr int kMaxSplitUnits = 40;        // (sequence, value head) pairs the split kernel takes
constexpr size_t kFlagBytesPerUnit = 128; // 16 ready flags + a consumed-chunk counter
constexpr size_t kRingOffset = 16384;
constexpr size_t kRingBytesPerUnit = 16 * 74752;  // record ring of one (sequence, value head)
static_assert(kFlagOffset + kMaxSplitUnits * kFlagBytesPerUnit <= kRingOffset, "workspace layout");

struct FwdParams {
  const void* q;         // [tokens, H, K]   io type
  const void* k;         // [tokens, H, K]   io type
  const void* v;         // [tokens, HV, V]  io type
  const float* g;        // [tokens, HV, K]
  const float* beta;     // [tokens, HV]
  const float* s0;       // [NS, HV, K, V] or null
  const int32_t* cu;     // [NS + 1] or null
  void* out;             // [tokens, HV, V]  io type
  float* sfin;           // [NS, HV, K, V] or null
  uint32_t* status;      // device status word
  uint8_t* ring;         // per-(sequence, value head) record ring (chunk kernel), or null
  unsigned long long wait_ns;  // limit of a bounded wait for work (drains have their own)
  // Pre-stage (kda_chunk_fwd_gated): 0 = inputs used as given; 1 = bounded gate, 2 =
  // softplus gate.  Then g_raw replaces g, beta holds raw values (sigmoid applied in
  // the kernel) and q, k are L2-normalised per row in the kernel.
  int prestage;
  const uint16_t* g_raw;  // [tokens, HV, K] bf16
  const float* A_log;     // [HV]
  const float* dt_bias;   // [HV, K]
  float lower_bound;      // bounded gate: g = lower_bound * sigmoid(exp(A_log) (g_raw + dt_bias))
  // State pass (kda_chunk_states): when h is set, the chains write the state entering
  // every chunk (bf16 [NS, HV, h_chunks, K, V]) and no output.
  uint16_t* h;
  int h_chunks;
  float scale;
  int T;                 // tokens per sequence (fixed length) or packed total
  int H, HV, K, V;
  int num_seqs;          // NS
  // Split chunk kernel: the launch takes the (sequence, value head) units [unit0, unit0 + NU)
  // of the sequence-major enumeration (larger problems run as several launches).
  int unit0;
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Token range [tok0, tok0 + len) of sequence `seq`.  With cu_seqlens each block
// checks the two entries it uses; a violation sets kStatusBounds and yields an
// empty range (the block then writes nothing).
__device__ __forceinline__ bool seq_range(const FwdParams& p, int seq, long& tok0, int& len) {
  if (p.cu == nullptr) {
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

}  // namespace kda
