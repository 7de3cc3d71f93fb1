// Forward kernel of fused scaled-dot-product attention for training
// (sdpfa_fwd of test_sdpa_loop_split, "DID loop split for SDPA", NVIDIA/Fuser
// PR 3711): out = dropout(softmax(scale * Q K^T + causal)) V and the
// natural-log log-sum-exp of each score row, stashed for the backward
// (NVIDIA/Fuser issue 2278, "SdpaOpFwd / SdpaOpBwd nodes").
//
// One CTA computes one 128-row query tile of one (batch, head):
//   warp 4      TMA producer: Q once, then K_j and V_j through a ring of
//               shared-memory stages (128-byte swizzled, 64-column slabs).
//   warp 5      TMEM allocator and MMA issuer (one thread): S_j = Q K_j^T
//               into one of two TMEM score buffers, then O += P_{j-1} V_{j-1}
//               so the tensor core computes the next scores while the
//               softmax warps work on the current ones.
//   warps 0-3   softmax: thread r owns query row r. It reads its score row
//               from TMEM, applies the causal / key-tail mask, keeps the
//               running row max m (base-2, scaled) and sum l, rescales the
//               O row in TMEM only when the max grew by more than 2^8,
//               writes P (bf16, dropout applied) to shared memory for the
//               P V product, and at the end writes out = O / l (TMA store)
//               and lse = (m + log2 l) * ln 2.
// Key tiles entirely above the causal diagonal are never loaded or computed.
#include "common.cuh"

namespace sdpa {
namespace {

template <int D>
struct FwdLayout {
  static constexpr int kSlabBytes = 128 * 128;            // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;          // 128 rows x D bf16
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;     // 128 x 128 bf16, 2 slabs
  static constexpr int kBar = kP + 2 * kSlabBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], s_empty[2], p_full, o_done, fin
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 3;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;             // room to align to 1024
  // TMEM columns
  static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemCols = 512;
};

__device__ __forceinline__ void reg_touch(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

template <int D, bool CAUSAL, bool DROPOUT>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdParams p) {
  using L = FwdLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + S;
  uint64_t* s_full = kv_empty + S;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* fin = o_done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int BH = p.B * p.H;
  int q_tile = blockIdx.x / BH;
  const int bh = blockIdx.x - q_tile * BH;
  if (CAUSAL) q_tile = p.n_q_tiles - 1 - q_tile;  // longest tiles first
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int q0 = q_tile * 128;
  int n_kv = (p.Sk + 127) / 128;
  if (CAUSAL) n_kv = min(n_kv, min(q0 + 127, p.Sq - 1) / 128 + 1);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(fin, 1);
    *abort_word = 0u;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_holder, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl wc{abort_word, p.err, p.wait_limit_ns};

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(q_full, L::kTileBytes);
#pragma unroll
      for (int s = 0; s < D / 64; ++s)
        tma_load_4d(smem + L::kQ + s * L::kSlabBytes, &tm_q, q_full, s * 64, q0, h, b);
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        if (j >= S) mbar_wait(&kv_empty[st], ((j / S) - 1) & 1, wc, kSiteFwdKvEmpty);
        mbar_arrive_expect_tx(&kv_full[st], 2 * L::kTileBytes);
#pragma unroll
        for (int s = 0; s < D / 64; ++s) {
          tma_load_4d(smem + L::kK + st * L::kTileBytes + s * L::kSlabBytes, &tm_k, &kv_full[st],
                      s * 64, j * 128, h, b);
          tma_load_4d(smem + L::kV + st * L::kTileBytes + s * L::kSlabBytes, &tm_v, &kv_full[st],
                      s * 64, j * 128, h, b);
        }
      }
      if (*abort_word) {
        // give the loads still in flight time to land before the CTA exits
        for (int j = max(0, n_kv - S); j < n_kv; ++j)
          mbar_wait_drain(&kv_full[j % S], (j / S) & 1, 2000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(128, D, false, true);
      const uint32_t tS[2] = {tmem + L::kTmemS0, tmem + L::kTmemS1};
      const uint32_t tO = tmem + L::kTmemO;
      mbar_wait(q_full, 0, wc, kSiteFwdQFull);
      for (int j = 0; j <= n_kv; ++j) {
        if (j < n_kv) {
          const int st = j % S;
          const int sbuf = j & 1;
          mbar_wait(&kv_full[st], (j / S) & 1, wc, kSiteFwdKvFull);
          if (j >= 2) mbar_wait(&s_empty[sbuf], ((j >> 1) - 1) & 1, wc, kSiteFwdSEmpty);
          tc_fence_after();
          const uint32_t qa = sb + L::kQ;
          const uint32_t ka = sb + L::kK + st * L::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * L::kSlabBytes + (kk & 3) * 32;
            mma_bf16_ss(tS[sbuf], sdesc_sw128(qa + koff, 16, 1024),
                        sdesc_sw128(ka + koff, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[sbuf]);
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int st = jj % S;
          mbar_wait(p_full, jj & 1, wc, kSiteFwdPFull);
          tc_fence_after();
          const uint32_t pa = sb + L::kP;
          const uint32_t va = sb + L::kV + st * L::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t poff = (kk >> 2) * L::kSlabBytes + (kk & 3) * 32;
            mma_bf16_ss(tO, sdesc_sw128(pa + poff, 16, 1024),
                        sdesc_sw128(va + kk * 2048, L::kSlabBytes, 1024), kIdO,
                        (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(o_done);
          mma_commit(&kv_empty[st]);
        }
      }
      // every MMA must be complete before the TMEM is released
      mma_commit(fin);
      mbar_wait_drain(fin, 0, 2000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int row = threadIdx.x;  // query row within the tile == TMEM lane
    const int qi = q0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS[2] = {tmem + L::kTmemS0 + lane_base, tmem + L::kTmemS1 + lane_base};
    const uint32_t tO = tmem + L::kTmemO + lane_base;
    const uint64_t n_row = (static_cast<uint64_t>(bh) * p.Sq + qi) * static_cast<uint64_t>(p.Sk);
    float m = -INFINITY;
    float l = 0.f;

    for (int j = 0; j < n_kv; ++j) {
      const int sbuf = j & 1;
      mbar_wait(&s_full[sbuf], (j >> 1) & 1, wc, kSiteFwdSFull);
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld32(tS[sbuf] + 0, r0);
      tmem_ld32(tS[sbuf] + 32, r1);
      tmem_ld32(tS[sbuf] + 64, r2);
      tmem_ld32(tS[sbuf] + 96, r3);
      tmem_ld_wait(r0);
      reg_touch(r1);
      reg_touch(r2);
      reg_touch(r3);
      tc_fence_before();
      mbar_arrive(&s_empty[sbuf]);

      float x[128];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = __uint_as_float(r0[i]) * p.scale_log2;
        x[32 + i] = __uint_as_float(r1[i]) * p.scale_log2;
        x[64 + i] = __uint_as_float(r2[i]) * p.scale_log2;
        x[96 + i] = __uint_as_float(r3[i]) * p.scale_log2;
      }
      const int k0 = j * 128;
      const bool tail = k0 + 128 > p.Sk;
      const bool diag = CAUSAL && (k0 + 127 > q0);
      if (tail || diag) {
        const int lim = CAUSAL ? min(p.Sk - k0, qi - k0 + 1) : (p.Sk - k0);
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) x[i] = -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int i = 1; i < 128; ++i) mx = fmaxf(mx, x[i]);
      const float m_new = fmaxf(m, mx);

      if (j >= 1) {
        // O and the P buffer are free once the previous P V product is done
        mbar_wait(o_done, (j - 1) & 1, wc, kSiteFwdODone);
        tc_fence_after();
        const bool grow = m_new > m + 8.0f;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = ex2_approx(m - m_new);
          l *= alpha;
          m = m_new;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + c * 32, o);
          }
          tmem_st_wait();
        }
      } else {
        m = m_new;
      }

      uint32_t keep[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (DROPOUT) keep_bits_128(n_row + k0, p.drop_threshold, p.pk, keep);
      float rs = 0.f;
      uint32_t pk2[64];
#pragma unroll
      for (int i = 0; i < 128; i += 2) {
        float e0 = ex2_approx(x[i] - m);
        float e1 = ex2_approx(x[i + 1] - m);
        rs += e0 + e1;
        if (DROPOUT) {
          e0 = ((keep[i >> 5] >> (i & 31)) & 1u) ? e0 * p.drop_rescale : 0.f;
          e1 = ((keep[(i + 1) >> 5] >> ((i + 1) & 31)) & 1u) ? e1 * p.drop_rescale : 0.f;
        }
        pk2[i >> 1] = pack_bf16x2(e0, e1);
      }
      l += rs;
      const uint32_t pa = sb + L::kP;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_shared_v4(pa + (c >> 3) * L::kSlabBytes + sw128_offset(row, c & 7), pk2[4 * c],
                     pk2[4 * c + 1], pk2[4 * c + 2], pk2[4 * c + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }

    // ------------------------------------------------------------ epilogue
    mbar_wait(o_done, (n_kv - 1) & 1, wc, kSiteFwdODone);
    tc_fence_after();
    const float inv_l = 1.f / l;
    const uint32_t oa = sb + L::kQ;  // Q is dead: every MMA has completed
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + c * 32, o);
      tmem_ld_wait(o);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int col0 = c * 32 + q4 * 8;
        const uint32_t addr = oa + (col0 >> 6) * L::kSlabBytes + sw128_offset(row, (col0 & 63) >> 3);
        st_shared_v4(addr,
                     pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l,
                                 __uint_as_float(o[q4 * 8 + 1]) * inv_l),
                     pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l,
                                 __uint_as_float(o[q4 * 8 + 3]) * inv_l),
                     pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l,
                                 __uint_as_float(o[q4 * 8 + 5]) * inv_l),
                     pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l,
                                 __uint_as_float(o[q4 * 8 + 7]) * inv_l));
      }
    }
    if (qi < p.Sq) p.lse[static_cast<size_t>(bh) * p.Sq + qi] = (m + log2f(l)) * kLn2;
    fence_async_smem();
    named_barrier_sync(1, 128);
    if (row == 0) {
#pragma unroll
      for (int s = 0; s < D / 64; ++s)
        tma_store_4d(&tm_o, smem + L::kQ + s * L::kSlabBytes, s * 64, q0, h, b);
      bulk_commit();
      bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, bool C, bool DR>
cudaError_t launch_fwd_t(const CUtensorMap* maps, const FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_kernel<D, C, DR>;
  const int smem = FwdLayout<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.n_q_tiles) * static_cast<unsigned>(p.B * p.H);
  kern<<<grid, 192, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int D) {
  return D == 64 ? FwdLayout<64>::kAlloc : FwdLayout<128>::kAlloc;
}

cudaError_t launch_fwd(int D, bool causal, bool dropout, const CUtensorMap* maps,
                       const FwdParams& p, cudaStream_t stream) {
#define SDPA_FWD_CASE(DD, CC, RR) \
  if (D == DD && causal == CC && dropout == RR) return launch_fwd_t<DD, CC, RR>(maps, p, stream);
  SDPA_FWD_CASE(64, false, false)
  SDPA_FWD_CASE(64, false, true)
  SDPA_FWD_CASE(64, true, false)
  SDPA_FWD_CASE(64, true, true)
  SDPA_FWD_CASE(128, false, false)
  SDPA_FWD_CASE(128, false, true)
  SDPA_FWD_CASE(128, true, false)
  SDPA_FWD_CASE(128, true, true)
#undef SDPA_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
