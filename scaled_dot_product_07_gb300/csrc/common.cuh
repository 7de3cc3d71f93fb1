// Kernel parameter blocks and constants shared by the attention kernels and
// their host-side launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "philox.cuh"
#include "ptx.cuh"

namespace sdpa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Codes written to the device error word when a bounded wait gives up
// (which role, which barrier).
enum WaitSite : uint32_t {
  kSiteFwdKvEmpty = 0x101, kSiteFwdQFull, kSiteFwdKvFull, kSiteFwdSEmpty, kSiteFwdPFull,
  kSiteFwdSFull, kSiteFwdODone,
  kSiteBwdKvFull = 0x201, kSiteBwdQFull, kSiteBwdQEmpty, kSiteBwdSpEmpty, kSiteBwdPFull,
  kSiteBwdDsFull, kSiteBwdDqEmpty, kSiteBwdSFull, kSiteBwdDpFull, kSiteBwdPdsEmpty,
  kSiteBwdDqFull, kSiteBwdDone,
  kSiteSelftest = 0x301,
};

struct FwdParams {
  int B, H, Sq, Sk;
  int n_q_tiles;          // ceil(Sq / 256): pairs of 128-row query tiles per head
  float scale_log2;       // softmax scale * log2(e)
  uint32_t drop_threshold;  // floor(p * 2^32)
  float drop_rescale;       // 1 / (1 - p)
  PhiloxKey pk;
  float* lse;             // [B, H, Sq] fp32
  uint32_t* err;          // device error word
  uint64_t wait_limit_ns;
};

struct BwdParams {
  int B, H, Sq, Sk, Sq_pad;
  int n_kv_tiles;         // ceil(Sk / 128)
  float scale_log2;
  float scale;
  uint32_t drop_threshold;
  float drop_rescale;
  PhiloxKey pk;
  float* dq_acc;          // workspace [B*H, Sq_pad, D] fp32
  const float* lse2;      // workspace [B*H, Sq_pad]: lse * log2(e), +inf past Sq
  const float* delta;     // workspace [B*H, Sq_pad]: rowsum(dO * O), 0 past Sq
  uint32_t* err;
  uint64_t wait_limit_ns;
};

// Strided bf16 [B,H,S,D] view used by the elementwise kernels.
struct StridedBf16 {
  void* data;
  int64_t sB, sH, sS;  // element strides (D is contiguous)
};

struct PreParams {
  int B, H, Sq, Sq_pad, D;
  StridedBf16 out, dout;
  const float* lse;       // [B,H,Sq]
  float* lse2;
  float* delta;
  float* dq_acc;
};

struct ConvParams {
  int B, H, Sq, Sq_pad, D;
  float scale;
  const float* dq_acc;
  StridedBf16 dq;
};

// Launchers (defined in the .cu files). Each returns the launch's CUDA error.
cudaError_t launch_fwd(int D, bool causal, bool dropout, const CUtensorMap* maps /*q,k,v,o*/,
                       const FwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const PreParams& p, cudaStream_t stream);
cudaError_t launch_bwd_main(int D, bool causal, bool dropout,
                            const CUtensorMap* maps /*q,k,v,do,dk,dv*/, const BwdParams& p,
                            cudaStream_t stream);
cudaError_t launch_bwd_main_d128(bool causal, bool dropout,
                                 const CUtensorMap* maps /*q,k,v,do,dk,dv*/, const BwdParams& p,
                                 cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(const ConvParams& p, cudaStream_t stream);
cudaError_t launch_zero_fill(StridedBf16 t, int B, int H, int S, int D, cudaStream_t stream);
cudaError_t launch_dropout_mask(int64_t B, int64_t H, int64_t Sq, int64_t Sk, uint32_t threshold,
                                PhiloxKey pk, uint8_t* mask, cudaStream_t stream);
cudaError_t launch_selftest_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t stream);

// Dynamic shared memory sizes (for validation against the device limit).
size_t fwd_smem_bytes(int D);
size_t bwd_smem_bytes(int D);
size_t bwd_d128_smem_bytes();

__host__ __device__ inline uint8_t* align_up_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023u) &
                                    ~static_cast<uintptr_t>(1023u));
}

}  // namespace sdpa
