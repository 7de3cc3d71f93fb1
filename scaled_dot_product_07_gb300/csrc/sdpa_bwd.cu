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
//   bwd_main_kernel        (head dim 64; head dim 128 has its own kernel in
//                          sdpa_bwd128.cu) one CTA per 128-key tile of one (batch, head); it
//                          walks the query tiles that can see its keys:
//                            S^T  = K Q_i^T             (tcgen05, TMEM)
//                            dP~^T = V dO_i^T           (tcgen05, TMEM)
//                            P^T  = exp2(S^T*scale*log2e - lse2_i), masked
//                            dV  += (P * keep/(1-p))^T dO_i
//                            dS^T = P^T * (dP~^T * keep/(1-p) - Delta_i)
//                            dK  += dS^T Q_i            (scale applied at the end)
//                            dQ_i partial = dS K       -> fp32 bulk reduce-add
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
        reinterpret_cast<const float4*>(p.dq_acc + (bh * p.Sq_pad + i) * p.D + part * 8);
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
    const float* src = p.dq_part + (bh * p.Sq_pad + i) * p.D + part * 8;
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

template <int D>
struct BwdLayout {
  static constexpr int kMq = 8192 / D;                  // query rows per step
  static constexpr int kKvBytes = 128 * D * 2;          // K or V tile
  static constexpr int kKvSlab = 128 * 128;             // 128 rows x 128 bytes
  static constexpr int kQSlab = kMq * 128;              // Mq rows x 128 bytes
  static constexpr int kQBytes = kMq * D * 2;           // Q or dO tile
  static constexpr int kStages = 2;
  static constexpr int kPtBytes = 128 * kMq * 2;        // [128 keys x Mq] bf16
  static constexpr int kPtSlab = 128 * 128;
  static constexpr int kDqBytes = kMq * D * 4;          // fp32 dQ staging
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKvBytes;
  static constexpr int kQ = kV + kKvBytes;
  static constexpr int kDO = kQ + kStages * kQBytes;
  static constexpr int kLse = kDO + kStages * kQBytes;
  static constexpr int kDelta = kLse + kStages * kMq * 4;
  static constexpr int kPt = kDelta + kStages * kMq * 4;
  static constexpr int kDst = kPt + kPtBytes;
  static constexpr int kDq = kDst + kPtBytes;
  static constexpr int kBar = kDq + kDqBytes;
  // kv_full, q_full[S], q_empty[S], s_full, dp_full, sp_empty, p_full, ds_full,
  // pds_empty, dq_full, dq_empty, done
  static constexpr int kNumBars = 1 + 2 * kStages + 9;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns
  static constexpr uint32_t kTmemDV = 0, kTmemDK = D, kTmemS = 2 * D, kTmemDP = 2 * D + kMq,
                            kTmemDQ = 2 * D + 2 * kMq, kTmemCols = 512;
  static_assert(kTmemDQ + 64 <= 512, "TMEM budget");
  static_assert(kKvBytes % 1024 == 0 && kQBytes % 1024 == 0 && (kLse % 1024) == 0, "align");
};

__device__ __forceinline__ void reg_touch32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

// Load kMq consecutive fp32 TMEM columns of this thread's lane into v[].
template <int N>
__device__ __forceinline__ void tmem_load_row(uint32_t taddr, float (&v)[N]) {
  static_assert(N == 64 || N == 128, "row width");
  uint32_t r0[32], r1[32];
  tmem_ld32(taddr, r0);
  tmem_ld32(taddr + 32, r1);
  if constexpr (N == 128) {
    uint32_t r2[32], r3[32];
    tmem_ld32(taddr + 64, r2);
    tmem_ld32(taddr + 96, r3);
    tmem_ld_wait(r0);
    reg_touch32(r1);
    reg_touch32(r2);
    reg_touch32(r3);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = __uint_as_float(r0[i]);
      v[32 + i] = __uint_as_float(r1[i]);
      v[64 + i] = __uint_as_float(r2[i]);
      v[96 + i] = __uint_as_float(r3[i]);
    }
  } else {
    tmem_ld_wait(r0);
    reg_touch32(r1);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = __uint_as_float(r0[i]);
      v[32 + i] = __uint_as_float(r1[i]);
    }
  }
}

// Write a row of N bf16 values (thread's row `row`) into a 128-byte-swizzled
// tile of 128-byte rows made of N/64 slabs of kPtSlab bytes.
template <int N>
__device__ __forceinline__ void store_row_bf16_sw128(uint32_t base, int row, const float (&v)[N]) {
#pragma unroll
  for (int c = 0; c < N / 8; ++c) {
    st_shared_v4(base + (c >> 3) * (128 * 128) + sw128_offset(row, c & 7),
                 pack_bf16x2(v[8 * c + 0], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                 pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
  }
}

template <int D, bool CAUSAL, bool DROPOUT, bool BIAS, bool VARLEN>
__global__ void __launch_bounds__(320, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const BwdParams p) {
  using L = BwdLayout<D>;
  constexpr int S = L::kStages;
  constexpr int MQ = L::kMq;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + S;
  uint64_t* s_full = q_empty + S;
  uint64_t* dp_full = s_full + 1;
  uint64_t* sp_empty = dp_full + 1;
  uint64_t* p_full = sp_empty + 1;
  uint64_t* ds_full = p_full + 1;
  uint64_t* pds_empty = ds_full + 1;
  uint64_t* dq_full = pds_empty + 1;
  uint64_t* dq_empty = dq_full + 1;
  uint64_t* done = dq_empty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // head-major order: the CTAs of one head run together, so the head's Q and
  // dO tiles (which every one of them streams) stay in L2; within a head the
  // low key tiles (the most causal work) go first
  const int slot = blockIdx.x / p.n_kv_tiles;
  const int kv_tile = blockIdx.x - slot * p.n_kv_tiles;
  // batch-major, or head-major when the bias is shared by the batch
  const int b = p.h_major ? slot % p.B : slot / p.H;
  const int h = p.h_major ? slot / p.B : slot - b * p.H;
  const int bh = b * p.H + h;
  const int k0 = kv_tile * 128;
  // the sequence: the whole [Sq, Sk] problem, or sequence b of a packed batch
  int Sq = p.Sq, Sk = p.Sk, qs = 0, ks = 0;
  if (VARLEN) {
    qs = p.cu_q[b];
    Sq = p.cu_q[b + 1] - qs;
    ks = p.cu_k[b];
    Sk = p.cu_k[b + 1] - ks;
    if (k0 >= Sk) return;  // no keys of the sequence in this tile
  }
  const int tb = VARLEN ? 0 : b;  // batch coordinate in the tensor maps
  const int n_qt = (Sq + MQ - 1) / MQ;
  const int qt_first = CAUSAL ? min(k0 / MQ, n_qt) : 0;
  const int n_steps = n_qt - qt_first;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(sp_empty, 128);
    mbar_init(p_full, 128);
    mbar_init(ds_full, 128);
    mbar_init(pds_empty, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(done, 1);
    *abort_word = 0u;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl wc{abort_word, p.err, p.wait_limit_ns};

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_steps > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * L::kKvBytes);
#pragma unroll
      for (int s = 0; s < D / 64; ++s) {
        tma_load_4d(smem + L::kK + s * L::kKvSlab, &tm_k, kv_full, s * 64, ks + k0, h, tb);
        tma_load_4d(smem + L::kV + s * L::kKvSlab, &tm_v, kv_full, s * 64, ks + k0, h, tb);
      }
      for (int t = 0; t < n_steps; ++t) {
        const int st = t % S;
        const int i0 = (qt_first + t) * MQ;
        if (t >= S) mbar_wait(&q_empty[st], ((t / S) - 1) & 1, wc, kSiteBwdQEmpty);
        mbar_arrive_expect_tx(&q_full[st], 2 * L::kQBytes + 2 * MQ * 4);
#pragma unroll
        for (int s = 0; s < D / 64; ++s) {
          tma_load_4d(smem + L::kQ + st * L::kQBytes + s * L::kQSlab, &tm_q, &q_full[st], s * 64,
                      qs + i0, h, tb);
          tma_load_4d(smem + L::kDO + st * L::kQBytes + s * L::kQSlab, &tm_do, &q_full[st],
                      s * 64, qs + i0, h, tb);
        }
        const size_t vec = static_cast<size_t>(bh) * p.Sq_pad + i0;
        bulk_load(smem + L::kLse + st * MQ * 4, p.lse2 + vec, MQ * 4, &q_full[st]);
        bulk_load(smem + L::kDelta + st * MQ * 4, p.delta + vec, MQ * 4, &q_full[st]);
      }
      if (*abort_word) {
        for (int t = max(0, n_steps - S); t < n_steps; ++t)
          mbar_wait_drain(&q_full[t % S], (t / S) & 1, 2000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and descriptor arithmetic are
    // warp-uniform); one elected lane issues the tcgen05 instructions.
    if (n_steps > 0) {
      const uint32_t leader = elect_one();
      constexpr uint32_t kIdSP = idesc_bf16_f32(128, MQ, false, false);   // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_bf16_f32(128, D, false, true);     // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, 64, true, true);      // dQ^T / dQ
      const uint32_t tS = tmem + L::kTmemS, tDP = tmem + L::kTmemDP;
      const uint32_t tDV = tmem + L::kTmemDV, tDK = tmem + L::kTmemDK, tDQ = tmem + L::kTmemDQ;
      const uint32_t ka = sb + L::kK, va = sb + L::kV, pa = sb + L::kPt, da = sb + L::kDst;
      mbar_wait(kv_full, 0, wc, kSiteBwdKvFull);
      for (int t = 0; t < n_steps; ++t) {
        const int st = t % S;
        const uint32_t qa = sb + L::kQ + st * L::kQBytes;
        const uint32_t oa = sb + L::kDO + st * L::kQBytes;
        mbar_wait(&q_full[st], (t / S) & 1, wc, kSiteBwdQFull);
        if (t >= 1) mbar_wait(sp_empty, (t - 1) & 1, wc, kSiteBwdSpEmpty);
        tc_fence_after();
        // S^T = K Q^T and dP~^T = V dO^T  (M = 128 keys, N = MQ, K = D)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kKvSlab + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * L::kQSlab + (kk & 3) * 32;
          mma_bf16_ss_if(leader, tS, sdesc_sw128(ka + koff, 16, 1024), sdesc_sw128(qa + qoff, 16, 1024),
                      kIdSP, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(leader, s_full);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kKvSlab + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * L::kQSlab + (kk & 3) * 32;
          mma_bf16_ss_if(leader, tDP, sdesc_sw128(va + koff, 16, 1024), sdesc_sw128(oa + qoff, 16, 1024),
                      kIdSP, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(leader, dp_full);
        // dV += P~^T dO  (M = 128 keys, N = D, K = MQ; dO read MN-major)
        mbar_wait(p_full, t & 1, wc, kSiteBwdPFull);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < MQ / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * L::kPtSlab + (kk & 3) * 32;
          mma_bf16_ss_if(leader, tDV, sdesc_sw128(pa + poff, 16, 1024),
                      sdesc_sw128(oa + kk * 2048, L::kQSlab, 1024), kIdKV,
                      (t > 0 || kk > 0) ? 1u : 0u);
        }
        // dK += dS^T Q
        mbar_wait(ds_full, t & 1, wc, kSiteBwdDsFull);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < MQ / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * L::kPtSlab + (kk & 3) * 32;
          mma_bf16_ss_if(leader, tDK, sdesc_sw128(da + poff, 16, 1024),
                      sdesc_sw128(qa + kk * 2048, L::kQSlab, 1024), kIdKV,
                      (t > 0 || kk > 0) ? 1u : 0u);
        }
        // dQ partial over this key tile (K = 128 keys); both operands MN-major.
        //   D = 128: dQ^T [D x MQ] = K^T dS^T   (A = K tile, B = dS^T tile)
        //   D =  64: dQ   [MQ x D] = dS K       (A = dS^T tile, B = K tile)
        if (t >= 1) mbar_wait(dq_empty, (t - 1) & 1, wc, kSiteBwdDqEmpty);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t kdesc = sdesc_sw128(ka + kk * 2048, L::kKvSlab, 1024);
          const uint64_t sdesc = sdesc_sw128(da + kk * 2048, L::kPtSlab, 1024);
          if constexpr (D == 128)
            mma_bf16_ss_if(leader, tDQ, kdesc, sdesc, kIdQ, kk > 0 ? 1u : 0u);
          else
            mma_bf16_ss_if(leader, tDQ, sdesc, kdesc, kIdQ, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(leader, dq_full);
        mma_commit_if(leader, &q_empty[st]);
        mma_commit_if(leader, pds_empty);
      }
      mma_commit_if(leader, done);
      mbar_wait_drain(done, 0, 2000000000ull);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ WG0: P^T and dS^T (thread = key)
    const int r = threadIdx.x;
    const int kj = k0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + L::kTmemS + lane_base, tDP = tmem + L::kTmemDP + lane_base;
    const uint32_t pa = sb + L::kPt, da = sb + L::kDst;
    const PhiloxKey pk = DROPOUT ? launch_key(p.pk, p.rng_dev) : p.pk;
    for (int t = 0; t < n_steps; ++t) {
      const int st = t % S;
      const int i0 = (qt_first + t) * MQ;
      const uint32_t lse_s = sb + L::kLse + st * MQ * 4;
      const uint32_t del_s = sb + L::kDelta + st * MQ * 4;
      const bool key_ok = kj < Sk;
      const uint16_t* bp = BIAS ? p.bias.data + b * p.bias.sB + h * p.bias.sH + (key_ok ? kj : 0)
                                : nullptr;
      // the step's dropout keep bits depend only on the indices: drawn while
      // the tensor core computes S^T
      uint32_t kb[MQ / 32];
#pragma unroll
      for (int w = 0; w < MQ / 32; ++w) kb[w] = 0xffffffffu;
      if (DROPOUT) {
        const uint64_t n_base = (counter_bh(b, h, p.b0, p.h0, p.H_total) * p.Sq_ctr + i0) *
                                    static_cast<uint64_t>(p.Sk_ctr) +
                                kj;
        if ((p.Sk_ctr & 3) == 0) {
          keep_bits_quad<MQ / 32>(n_base, static_cast<uint64_t>(p.Sk_ctr), p.drop_threshold, pk,
                                  kb);
        } else {
#pragma unroll
          for (int c = 0; c < MQ; ++c) {
            const bool kp =
                keep_one(n_base + static_cast<uint64_t>(c) * p.Sk_ctr, p.drop_threshold, pk);
            if (!kp) kb[c >> 5] &= ~(1u << (c & 31));
          }
        }
      }
      mbar_wait(&q_full[st], (t / S) & 1, wc, kSiteBwdQFull);
      mbar_wait(s_full, t & 1, wc, kSiteBwdSFull);
      tc_fence_after();
      float pv[MQ];
      tmem_load_row<MQ>(tS, pv);
      const bool need_mask = (k0 + 128 > Sk) || (CAUSAL && i0 < k0 + 127);
      // visible query rows of this key: qi >= kj (causal) and the key exists
      const int first_vis = kj >= Sk ? (1 << 30) : (CAUSAL ? kj - i0 : 0);
#pragma unroll
      for (int cc = 0; cc < MQ / 32; ++cc) {
        uint32_t bpk[16];  // bias of query rows i0 + 32cc .. +32 at key kj, bf16 pairs
        if (BIAS) {
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            const int ia = i0 + 32 * cc + 2 * c2;
            const uint32_t lo =
                (key_ok && ia < Sq) ? __ldg(bp + static_cast<int64_t>(ia) * p.bias.sS) : 0u;
            const uint32_t hi = (key_ok && ia + 1 < Sq)
                                    ? __ldg(bp + static_cast<int64_t>(ia + 1) * p.bias.sS)
                                    : 0u;
            bpk[c2] = lo | (hi << 16);
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = 32 * cc + i;
          float arg = fmaf(pv[c], p.scale_log2, -ld_shared_f32(lse_s + c * 4));
          if (BIAS)
            arg = fmaf(bf16_bits_to_float((i & 1) ? (bpk[i >> 1] >> 16) : (bpk[i >> 1] & 0xffffu)),
                       kLog2e, arg);
          float e = ex2_approx(arg);
          if (need_mask && c < first_vis) e = 0.f;
          pv[c] = e;
        }
      }
      if (t >= 1) mbar_wait(pds_empty, (t - 1) & 1, wc, kSiteBwdPdsEmpty);
#pragma unroll
      for (int c = 0; c < MQ / 8; ++c) {
        float q8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = 8 * c + k;
          q8[k] = DROPOUT ? (((kb[e >> 5] >> (e & 31)) & 1u) ? pv[e] * p.drop_rescale : 0.f) : pv[e];
        }
        st_shared_v4(pa + (c >> 3) * L::kPtSlab + sw128_offset(r, c & 7), pack_bf16x2(q8[0], q8[1]),
                     pack_bf16x2(q8[2], q8[3]), pack_bf16x2(q8[4], q8[5]), pack_bf16x2(q8[6], q8[7]));
      }
      fence_async_smem();
      mbar_arrive(p_full);

      mbar_wait(dp_full, t & 1, wc, kSiteBwdDpFull);
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < MQ / 32; ++cc) {
        uint32_t d[32];
        tmem_ld32(tDP + cc * 32, d);
        tmem_ld_wait(d);
        float ds[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = cc * 32 + i;
          float g = __uint_as_float(d[i]);
          if (DROPOUT) g = ((kb[cc] >> i) & 1u) ? g * p.drop_rescale : 0.f;
          ds[i] = pv[e] * (g - ld_shared_f32(del_s + e * 4));
        }
        if (BIAS && p.dbias.data != nullptr && key_ok) {
          // dbias(i, kj) = dS(i, kj); a warp writes 64 contiguous bytes per row
          uint16_t* dp = p.dbias.data + b * p.dbias.sB + h * p.dbias.sH + kj;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int qi = i0 + cc * 32 + i;
            if (qi < Sq)
              dp[static_cast<int64_t>(qi) * p.dbias.sS] =
                  static_cast<uint16_t>(pack_bf16x2(ds[i], 0.f) & 0xffffu);
          }
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c = cc * 4 + q4;  // 16-byte chunk index along the row
          st_shared_v4(da + (c >> 3) * L::kPtSlab + sw128_offset(r, c & 7),
                       pack_bf16x2(ds[8 * q4 + 0], ds[8 * q4 + 1]), pack_bf16x2(ds[8 * q4 + 2], ds[8 * q4 + 3]),
                       pack_bf16x2(ds[8 * q4 + 4], ds[8 * q4 + 5]), pack_bf16x2(ds[8 * q4 + 6], ds[8 * q4 + 7]));
        }
      }
      tc_fence_before();
      mbar_arrive(sp_empty);  // S^T and dP^T have been read
      fence_async_smem();
      mbar_arrive(ds_full);
    }
  } else {
    // ------------------------------------------------------------ WG1: dQ readout (warps 4-7)
    const int lt = threadIdx.x - 128;  // TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const uint32_t tDQ = tmem + L::kTmemDQ + lane_base;
    const uint32_t qa = sb + L::kDq;
    float* part = p.dq_part ? p.dq_part + static_cast<size_t>(kv_tile) * p.part_stride : nullptr;
    for (int t = 0; t < n_steps; ++t) {
      const int i0 = (qt_first + t) * MQ;
      mbar_wait(dq_full, t & 1, wc, kSiteBwdDqFull);
      tc_fence_after();
      float v[64];
      tmem_load_row<64>(tDQ, v);
      tc_fence_before();
      mbar_arrive(dq_empty);
      if (lt == 0) bulk_wait_read_all();  // the previous reduce has read the staging tile
      named_barrier_sync(2, 128);
      if constexpr (D == 128) {
        // lane = d, columns = query rows; staging is row-major [MQ][D] fp32
#pragma unroll
        for (int c = 0; c < 64; ++c) st_shared_f32(qa + (c * D + lt) * 4, v[c]);
      } else {
        // lane = query row, columns = d: 16 chunks of 4 floats per 256-byte row.
        // Rotating the chunk order by (row & 7) spreads the 8 rows of each
        // quarter-warp store over all banks.
        const int rot = lt & 7;
        float4 ch[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) ch[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
#pragma unroll
        for (int bit = 0; bit < 3; ++bit) {
          const bool on = (rot >> bit) & 1;
          float4 tmp[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) tmp[c] = on ? ch[(c + (1 << bit)) & 15] : ch[c];
#pragma unroll
          for (int c = 0; c < 16; ++c) ch[c] = tmp[c];
        }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_shared_v4f(qa + lt * 256 + ((c + rot) & 15) * 16, ch[c].x, ch[c].y, ch[c].z, ch[c].w);
      }
      fence_async_smem();
      named_barrier_sync(2, 128);
      if (lt == 0) {
        dq_out(p.dq_acc, part, (static_cast<size_t>(bh) * p.Sq_pad + i0) * D, smem + L::kDq,
               L::kDqBytes);
        bulk_commit();
      }
    }
    if (lt == 0) bulk_wait_all();
  }

  // ------------------------------------------------------------ epilogue: dK, dV
  if (warp < 8) {
    const bool is_dv = warp < 4;
    const int r = threadIdx.x & 127;
    const int wq = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t acc = tmem + (is_dv ? L::kTmemDV : L::kTmemDK) + lane_base;
    const uint32_t stage = sb + (is_dv ? L::kK : L::kV);  // K/V tiles are dead after `done`
    const float mul = is_dv ? 1.f : p.scale;
    // a packed sequence's last key tile is stored row by row, so that rows
    // of the next sequence are never written (uniform over the CTA)
    const bool direct = VARLEN && (k0 + 128 > Sk);
    if (n_steps > 0) {
      mbar_wait(done, 0, wc, kSiteBwdDone);
      tc_fence_after();
    }
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float v[32];
      if (n_steps > 0) {
        uint32_t o[32];
        tmem_ld32(acc + c * 32, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * mul;
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int col0 = c * 32 + q4 * 8;
        const uint32_t w0 = pack_bf16x2(v[q4 * 8 + 0], v[q4 * 8 + 1]);
        const uint32_t w1 = pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]);
        const uint32_t w2 = pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]);
        const uint32_t w3 = pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]);
        if (direct) {
          if (k0 + r < Sk && col0 < p.D_io) {
            const StridedBf16& o = is_dv ? p.dv_io : p.dk_io;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(o.data) + h * o.sH +
                                      static_cast<int64_t>(ks + k0 + r) * o.sS + col0) =
                make_uint4(w0, w1, w2, w3);
          }
        } else {
          st_shared_v4(stage + (col0 >> 6) * L::kKvSlab + sw128_offset(r, (col0 & 63) >> 3), w0,
                       w1, w2, w3);
        }
      }
    }
    if (!direct) {
      fence_async_smem();
      named_barrier_sync(is_dv ? 3 : 4, 128);
      if (r == 0) {
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_store_4d(is_dv ? &tm_dv : &tm_dk, smem + (is_dv ? L::kK : L::kV) + s * L::kKvSlab,
                       s * 64, ks + k0, h, tb);
        bulk_commit();
        bulk_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, bool C, bool DR, bool BI, bool VL>
cudaError_t launch_bwd_t(const CUtensorMap* m, const BwdParams& p, cudaStream_t stream) {
  auto kern = bwd_main_kernel<D, C, DR, BI, VL>;
  const int smem = BwdLayout<D>::kAlloc;
  cudaError_t e = ensure_smem_attr<bwd_main_kernel<D, C, DR, BI, VL>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.n_kv_tiles) * static_cast<unsigned>(p.B * p.H);
  kern<<<grid, 320, smem, stream>>>(m[0], m[1], m[2], m[3], m[4], m[5], p);
  return cudaGetLastError();
}

unsigned elementwise_grid(int64_t work_items) {
  const int64_t blocks = (work_items + 255) / 256;
  return static_cast<unsigned>(blocks < 1 ? 1 : (blocks > 152 * 16 ? 152 * 16 : blocks));
}

}  // namespace

size_t bwd_smem_bytes(int D) {
  return D == 64 ? BwdLayout<64>::kAlloc : bwd_d128_smem_bytes();
}

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
  const bool bias = p.bias.data != nullptr;
  const bool varlen = p.cu_q != nullptr;  // packed batches take no bias
#define SDPA_BWD_CASE(DD, CC, RR)                                                    \
  if (D == DD && causal == CC && dropout == RR)                                      \
    return varlen ? launch_bwd_t<DD, CC, RR, false, true>(maps, p, stream)           \
                  : (bias ? launch_bwd_t<DD, CC, RR, true, false>(maps, p, stream)   \
                          : launch_bwd_t<DD, CC, RR, false, false>(maps, p, stream));
  SDPA_BWD_CASE(64, false, false)
  SDPA_BWD_CASE(64, false, true)
  SDPA_BWD_CASE(64, true, false)
  SDPA_BWD_CASE(64, true, true)
#undef SDPA_BWD_CASE
  if (D == 128) return launch_bwd_main_d128(causal, dropout, maps, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
