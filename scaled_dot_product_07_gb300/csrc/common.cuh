// Kernel parameter blocks and constants shared by the attention kernels and
// their host-side launchers.
#pragma once

#include <atomic>
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
  kSiteFwdSFull, kSiteFwdODone, kSiteFwdBiasFull, kSiteFwdBiasEmpty,
  kSiteBwdKvFull = 0x201, kSiteBwdQFull, kSiteBwdQEmpty, kSiteBwdSpEmpty, kSiteBwdPFull,
  kSiteBwdDsFull, kSiteBwdDqEmpty, kSiteBwdSFull, kSiteBwdDpFull, kSiteBwdPdsEmpty,
  kSiteBwdDqFull, kSiteBwdDone,
  kSiteSelftest = 0x301,
};

// Strided bf16 [B,H,S,D] view used by the elementwise kernels.
struct StridedBf16 {
  void* data;
  int64_t sB, sH, sS;  // element strides (D is contiguous)
};

// Additive attention bias: bf16 [B or 1, H or 1, Sq, Sk], keys contiguous;
// a shared (size-1) batch or head dim has stride 0.
struct AttnBias {
  const uint16_t* data;       // bf16 bits; null: no bias
  int64_t sB, sH, sS;         // element strides
};

// Gradient of the bias, bf16 [B, H, Sq, Sk], keys contiguous (null: not wanted).
struct DBias {
  uint16_t* data;
  int64_t sB, sH, sS;
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

struct FwdParams {
  int B, H, Sq, Sk;
  int n_q_tiles;          // ceil(Sq / 256): pairs of 128-row query tiles per head
  float scale_log2;       // softmax scale * log2(e)
  uint32_t drop_threshold;  // floor(p * 2^32)
  float drop_rescale;       // 1 / (1 - p)
  int two_items;            // CTAs run items c and total-1-c (else one item each)
  PhiloxKey pk;
  PhiloxRoundKeys rk;       // round keys of pk.k0, pk.k1 (used when rng_dev is null)
  const uint64_t* rng_dev;  // device {seed, offset} overriding pk, or null
  int b0, h0, H_total;      // counter position of this launch in the whole problem
  AttnBias bias;
  float bias_to_raw;        // 1 / scale
  int h_major;              // CTA order by head, then batch (a batch-shared bias stays in L2)
  // packed variable-length batches (null: one [Sq, Sk] problem per (b, h)):
  // sequence b is query rows [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1])
  const int32_t* cu_q;
  const int32_t* cu_k;
  int Sq_ctr, Sk_ctr;       // dims of the dropout counter (Sq, Sk; or the max lengths)
  int total_q;              // packed query rows (lse is [H, total_q] when packed)
  // dropout keep bits stored for the backward (null: not stored): word
  // (bh*bits_kw + w)*bits_rows + i holds keys 32w .. 32w+31 of row i
  uint32_t* drop_bits;
  int64_t bits_kw, bits_rows;
  int D_io;                 // the caller's head dim (columns of out)
  StridedBf16 out_io;       // out, for the direct stores of a sequence's last tile
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
  const uint64_t* rng_dev;
  int b0, h0, H_total;
  AttnBias bias;
  DBias dbias;
  int h_major;
  // packed variable-length batches (null: one [Sq, Sk] problem per (b, h))
  const int32_t* cu_q;
  const int32_t* cu_k;
  int Sq_ctr, Sk_ctr;       // dims of the dropout counter
  // dropout keep bits the forward stored (null: drawn here), laid out as in
  // FwdParams
  const uint32_t* drop_bits;
  int64_t bits_kw, bits_rows;
  int D_io;                 // the caller's head dim (columns of dk, dv)
  StridedBf16 dk_io, dv_io; // for the direct stores of a sequence's last key tile
  StridedBf16 k_io;         // k, read row by row by the 256-wide kernel (K into TMEM)
  int acc_w;              // dQ accumulator row width: 64 when D <= 64, else 128
  float* dq_acc;          // workspace [B*H, Sq_pad, D] fp32 (reduce-add), or
  float* dq_part;         // deterministic mode: [n_kv_tiles][B*H, Sq_pad, D] fp32,
  size_t part_stride;     // one plain-stored partial per key tile (floats per slice)
  const float* lse2;      // workspace [B*H, Sq_pad]: lse * log2(e), +inf past Sq
  const float* delta;     // workspace [B*H, Sq_pad]: rowsum(dO * O), 0 past Sq
  uint32_t* err;
  uint64_t wait_limit_ns;
};


// D is the backward kernel's head dim (128 or 256: the width of the fp32 dQ rows);
// D_io the caller's head dim (a multiple of 8, at most D), the width of the
// rows read from out / dout and written to dq.
struct PreParams {
  int B, H, Sq, Sq_pad, D, D_io;
  const int32_t* cu_q;    // packed batch: sequence b's rows (Sq is then the maximum length)
  int total_q;
  StridedBf16 out, dout;
  const float* lse;       // [B,H,Sq]
  float* lse2;
  float* delta;
  float* dq_acc;          // zeroed here; null when the dQ partials are stored instead
};

struct ConvParams {
  int B, H, Sq, Sq_pad, D, D_io;
  const int32_t* cu_q;
  float scale;
  const float* dq_acc;
  StridedBf16 dq;
};

// Deterministic dQ: dq = scale * sum over the key tiles that see the row, in
// key-tile order, of the stored partials.
struct SumParams {
  int B, H, Sq, Sq_pad, D, D_io;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int n_kv_tiles;
  int causal;
  float scale;
  const float* dq_part;
  size_t part_stride;
  StridedBf16 dq;
};

// Float offset of element (row i, column c) of (batch, head) bh in the fp32
// dQ accumulator (or one deterministic-mode slice) of width D (64 for head
// dims up to 64, else the backward kernel's 128 or 256): the columns are
// split into blocks of w = min(D, 128) = 2^sh, and each block's rows are
// contiguous, [B*H][D/w][Sq_pad][w] (plain rows at D = 64 and 128).
__host__ __device__ __forceinline__ size_t dq_acc_offset(int64_t bh, int64_t i, int c, int D,
                                                        int Sq_pad) {
  const int sh = D == 64 ? 6 : 7;
  return (((static_cast<size_t>(bh) * (D >> sh) + (c >> sh)) * Sq_pad + i) << sh) +
         (c & ((1 << sh) - 1));
}

// Opt the kernel into `bytes` of dynamic shared memory, once per device: later
// launches (including those recorded while a stream is being captured into a
// CUDA graph) then make no call besides the launch itself.
template <auto Kern>
cudaError_t ensure_smem_attr(int bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// SMs of the current device, queried once per device (0 on error).
inline int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool cached = dev >= 0 && dev < 64;
  if (cached) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cached) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Launchers (defined in the .cu files). Each returns the launch's CUDA error.
cudaError_t launch_fwd(int D, bool causal, bool dropout, const CUtensorMap* maps /*q,k,v,o*/,
                       const FwdParams& p, cudaStream_t stream);
// The forward for head dims 136..256: one 128-row query tile per CTA
// (p.n_q_tiles = ceil(Sq / 128)); maps q (box 64 x 128 rows), k, v (64 x 64).
cudaError_t launch_fwd_d256(bool causal, bool dropout, const CUtensorMap* maps /*q,k,v*/,
                            const FwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const PreParams& p, cudaStream_t stream);
cudaError_t launch_bwd_dq_sum(const SumParams& p, cudaStream_t stream);
cudaError_t launch_bwd_main(int D, bool causal, bool dropout,
                            const CUtensorMap* maps /*q,k,v,do,dk,dv,bias,dbias,dq*/, const BwdParams& p,
                            cudaStream_t stream);
cudaError_t launch_bwd_main_d128(bool causal, bool dropout,
                                 const CUtensorMap* maps /*q,k,v,do,dk,dv,bias,dbias,dq*/, const BwdParams& p,
                                 cudaStream_t stream);
// The backward for kernel head dim 256: two CTAs (column halves) per 128-key
// tile; maps q, dout (box 64 x 32 rows), k, v, dk, dv (64 x 128).
cudaError_t launch_bwd_main_d256(bool causal, bool dropout,
                                 const CUtensorMap* maps /*q,k,v,do,dk,dv*/, const BwdParams& p,
                                 cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(const ConvParams& p, cudaStream_t stream);
cudaError_t launch_zero_fill(StridedBf16 t, int B, int H, int S, int D, cudaStream_t stream);
// Zeroes dbias(i, j) for j >= 128 * (i / 128 + 1): the key tiles a causal
// backward never visits for row i.
cudaError_t launch_dbias_zero_causal(const DBias& t, int B, int H, int Sq, int Sk,
                                     cudaStream_t stream);

}  // namespace sdpa
