// Backward of fused scaled-dot-product attention (sdpfa_bwd of
// test_sdpa_loop_split, "DID loop split for SDPA", NVIDIA/Fuser PR 3711):
// q_grad, k_grad, v_grad from out_grad, q, k, v, attn, log_sumexp and the
// dropout state (seed, offset). The probabilities are recomputed from the
// stashed log-sum-exp instead of being stored (NVIDIA/Fuser issue 2278,
// "stash vs recompute"); the dropout mask is regenerated from the absolute
// element index ("REDO of dropout support for mem eff #102038").
//
// Three kernels on one stream:
//   bwd_preprocess_kernel  Delta_i = sum_e dO_ie * O_ie, lse * log2(e) into a
//                          padded workspace (+inf past Sq), dQ accumulator := 0
//   main kernel            (sdpa_bwd128.cu for head dims up to 128 on 128-wide
//                          tiles, sdpa_bwd256.cu above)
//                          one CTA per 128-key tile of one (batch, head); it
//                          walks the query steps that can see its keys and
//                          reduce-adds each step's fp32 dQ partial
//   bwd_dq_convert_kernel  dq = scale * dQ accumulator -> bf16, caller layout
#include "common.cuh"

namespace sdpa {
namespace {

// ---------------------------------------------------------------- preprocess

__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const PreParams p) {
  const int tpr = p.D / 8;  // threads per row, 8 elements (16 bytes) each
  const int64_t total = static_cast<int64_t>(p.B) * p.H * p.Sq_pad;
  const int part = threadIdx.x % tpr;
  const int64_t row_step = static_cast<int64_t>(gridDim.x) * (blockDim.x / tpr);
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / tpr;
       row < total; row += row_step) {
    const int64_t bh = row / p.Sq_pad;
    const int i = static_cast<int>(row - bh * p.Sq_pad);
    const int b = static_cast<int>(bh / p.H);
    const int h = static_cast<int>(bh - static_cast<int64_t>(b) * p.H);
    // row i of sequence b: the problem's row, or packed row qs + i
    int len = p.Sq, qs = 0, tb = b;
    if (p.cu_q != nullptr) {
      qs = p.cu_q[b];
      len = p.cu_q[b + 1] - qs;
      tb = 0;
    }
    float acc = 0.f;
    if (i < len && part * 8 < p.D_io) {  // columns past D_io are the kernels' zero padding
      const int64_t eo = tb * p.out.sB + h * p.out.sH + static_cast<int64_t>(qs + i) * p.out.sS + part * 8;
      const int64_t ed =
          tb * p.dout.sB + h * p.dout.sH + static_cast<int64_t>(qs + i) * p.dout.sS + part * 8;
      const uint4 o = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.out.data) + eo);
      const uint4 d = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout.data) + ed);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&d);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 of = __bfloat1622float2(o2[k]);
        const float2 df = __bfloat1622float2(d2[k]);
        acc = fmaf(of.x, df.x, acc);
        acc = fmaf(of.y, df.y, acc);
      }
    }
    // groups of tpr consecutive lanes hold one row
    for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (p.dq_acc != nullptr) {
      float4* z = reinterpret_cast<float4*>(p.dq_acc + row * p.D + part * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (part == 0) {
      p.delta[row] = acc;
      const size_t li = p.cu_q != nullptr ? static_cast<size_t>(h) * p.total_q + qs + i
                                          : static_cast<size_t>(bh) * p.Sq + i;
      p.lse2[row] = i < len ? p.lse[li] * kLog2e : INFINITY;
    }
  }
}

// ---------------------------------------------------------------- dQ convert

__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const ConvParams p) {
  const int cpr = p.D_io / 8;  // 8-element chunks per output row
  const int64_t total = static_cast<int64_t>(p.B) * p.H * p.Sq * cpr;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = idx / cpr;
    const int part = static_cast<int>(idx - row * cpr);
    const int64_t bh = row / p.Sq;
    const int i = static_cast<int>(row - bh * p.Sq);
    const int b = static_cast<int>(bh / p.H);
    const int h = static_cast<int>(bh - static_cast<int64_t>(b) * p.H);
    int qs = 0, tb = b;
    if (p.cu_q != nullptr) {  // packed: rows past the sequence's length do not exist
      qs = p.cu_q[b];
      if (i >= p.cu_q[b + 1] - qs) continue;
      tb = 0;
    }
    const float4* src =
        reinterpret_cast<const float4*>(p.dq_acc + dq_acc_offset(bh, i, part * 8, p.D, p.Sq_pad));
    const float4 a = src[0], c = src[1];
    uint4 o;
    o.x = pack_bf16x2(a.x * p.scale, a.y * p.scale);
    o.y = pack_bf16x2(a.z * p.scale, a.w * p.scale);
    o.z = pack_bf16x2(c.x * p.scale, c.y * p.scale);
    o.w = pack_bf16x2(c.z * p.scale, c.w * p.scale);
    const int64_t e = tb * p.dq.sB + h * p.dq.sH + static_cast<int64_t>(qs + i) * p.dq.sS + part * 8;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq.data) + e) = o;
  }
}

// ---------------------------------------------------------------- deterministic dQ sum

// Key tile k stores a partial for every query row r >= 128 k (causal, top-left;
// every row otherwise): the sum runs over exactly those tiles, in tile order,
// so the result does not depend on the order in which the CTAs finished.
__global__ void __launch_bounds__(256) bwd_dq_sum_kernel(const SumParams p) {
  const int cpr = p.D_io / 8;
  const int64_t total = static_cast<int64_t>(p.B) * p.H * p.Sq * cpr;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = idx / cpr;
    const int part = static_cast<int>(idx - row * cpr);
    const int64_t bh = row / p.Sq;
    const int i = static_cast<int>(row - bh * p.Sq);
    const int b = static_cast<int>(bh / p.H);
    const int h = static_cast<int>(bh - static_cast<int64_t>(b) * p.H);
    int qs = 0, tb = b, n_kv = p.n_kv_tiles;
    if (p.cu_q != nullptr) {  // packed: this sequence's rows and key tiles only
      qs = p.cu_q[b];
      if (i >= p.cu_q[b + 1] - qs) continue;
      n_kv = (p.cu_k[b + 1] - p.cu_k[b] + 127) / 128;
      tb = 0;
    }
    const int k_last = p.causal ? min(n_kv - 1, i / 128) : n_kv - 1;
    const float* src = p.dq_part + dq_acc_offset(bh, i, part * 8, p.D, p.Sq_pad);
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k <= k_last; ++k) {
      const float4* s4 = reinterpret_cast<const float4*>(src + static_cast<size_t>(k) * p.part_stride);
      const float4 x = s4[0], y = s4[1];
      a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
      a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
    }
    uint4 o;
    o.x = pack_bf16x2(a[0] * p.scale, a[1] * p.scale);
    o.y = pack_bf16x2(a[2] * p.scale, a[3] * p.scale);
    o.z = pack_bf16x2(a[4] * p.scale, a[5] * p.scale);
    o.w = pack_bf16x2(a[6] * p.scale, a[7] * p.scale);
    const int64_t e = tb * p.dq.sB + h * p.dq.sH + static_cast<int64_t>(qs + i) * p.dq.sS + part * 8;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq.data) + e) = o;
  }
}

// One warp per dbias row i: zeroes keys [128 (i/128 + 1), Sk), which no key
// tile of a causal backward writes for that row.
__global__ void __launch_bounds__(256) dbias_zero_causal_kernel(DBias t, int B, int H, int Sq,
                                                                int Sk) {
  const int64_t rows = static_cast<int64_t>(B) * H * Sq;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; row < rows;
       row += warps) {
    const int64_t bh = row / Sq;
    const int i = static_cast<int>(row - bh * Sq);
    const int b = static_cast<int>(bh / H);
    const int h = static_cast<int>(bh - static_cast<int64_t>(b) * H);
    uint16_t* r = t.data + b * t.sB + h * t.sH + static_cast<int64_t>(i) * t.sS;
    for (int j = 128 * (i / 128 + 1) + lane; j < Sk; j += 32) r[j] = 0;
  }
}

__global__ void __launch_bounds__(256) zero_fill_kernel(StridedBf16 t, int B, int H, int S, int D) {
  const int cpr = D / 8;
  const int64_t total = static_cast<int64_t>(B) * H * S * cpr;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = idx / cpr;
    const int part = static_cast<int>(idx - row * cpr);
    const int64_t bh = row / S;
    const int i = static_cast<int>(row - bh * S);
    const int b = static_cast<int>(bh / H);
    const int h = static_cast<int>(bh - static_cast<int64_t>(b) * H);
    const int64_t e = b * t.sB + h * t.sH + i * t.sS + part * 8;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(t.data) + e) = make_uint4(0, 0, 0, 0);
  }
}

// ---------------------------------------------------------------- main kernel

// Grid of the grid-stride elementwise kernels: 256 threads per block, at
// most 16 blocks per SM of a 152-SM GPU.
unsigned elementwise_grid(int64_t work_items) {
  const int64_t blocks = (work_items + 255) / 256;
  return static_cast<unsigned>(blocks < 1 ? 1 : (blocks > 152 * 16 ? 152 * 16 : blocks));
}

}  // namespace

cudaError_t launch_bwd_preprocess(const PreParams& p, cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(p.B) * p.H * p.Sq_pad * (p.D / 8);
  bwd_preprocess_kernel<<<elementwise_grid(threads), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(const ConvParams& p, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.B) * p.H * p.Sq * (p.D_io / 8);
  bwd_dq_convert_kernel<<<elementwise_grid(items), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_sum(const SumParams& p, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.B) * p.H * p.Sq * (p.D_io / 8);
  bwd_dq_sum_kernel<<<elementwise_grid(items), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dbias_zero_causal(const DBias& t, int B, int H, int Sq, int Sk,
                                     cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(B) * H * Sq;
  if (rows == 0 || Sk == 0) return cudaSuccess;
  dbias_zero_causal_kernel<<<elementwise_grid(rows * 32), 256, 0, stream>>>(t, B, H, Sq, Sk);
  return cudaGetLastError();
}

cudaError_t launch_zero_fill(StridedBf16 t, int B, int H, int S, int D, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(B) * H * S * (D / 8);
  if (items == 0) return cudaSuccess;
  zero_fill_kernel<<<elementwise_grid(items), 256, 0, stream>>>(t, B, H, S, D);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(int D, bool causal, bool dropout, const CUtensorMap* maps,
                            const BwdParams& p, cudaStream_t stream) {
  // head dims up to 128 run the 128-wide kernel (sdpa_bwd128.cu), larger ones
  // the 256-wide kernel (sdpa_bwd256.cu)
  if (D == 128) return launch_bwd_main_d128(causal, dropout, maps, p, stream);
  if (D == 256) return launch_bwd_main_d256(causal, dropout, maps, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
