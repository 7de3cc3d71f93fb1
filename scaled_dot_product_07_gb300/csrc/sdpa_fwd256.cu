// Forward kernel of fused scaled-dot-product attention for head dims 136..256
// (kernel width 256; the caller's columns past D are read as zeros by TMA and
// never stored). Same operation as the narrower forward (sdpfa_fwd of
// test_sdpa_loop_split, "DID loop split for SDPA", NVIDIA/Fuser PR 3711):
// out = dropout(softmax(scale * Q K^T + causal)) V and the natural-log
// log-sum-exp of each score row.
//
// At D = 256 a 128-row query tile is 64 KB of bf16 and its O accumulator
// fills 256 of the 512 TMEM columns, so a CTA holds one query tile and
// streams 64-key K and V tiles (32 KB each) through one 5-slot ring in the
// order K_0, V_0, K_1, V_1, ... (Q 64 KB + 160 KB of shared memory); a slot
// is refilled once the product that reads it is done. 320 threads:
//   warp 9      TMA producer: Q once, then K_j and V_j into the ring.
//   warp 8      TMEM allocator and MMA issuer (converged warp, one elected
//               lane issues). TMEM: S[2] (64 fp32 columns each, by key-tile
//               parity) and O (256 columns). Per key tile j it issues
//                 S_{j+1} = Q K_{j+1}^T,  then  O += P_j V_j,
//               so the scores of the next tile are computed while the
//               softmax works on this one. P_j is bf16, written by the
//               softmax into the first 32 columns of S[j&1] and read from
//               TMEM as the A operand.
//   warps 0-7   softmax: thread (half, r) owns keys [32 half, 32 half + 32)
//               of query row r of each 64-key tile (warps w and w+4 share
//               TMEM lanes); the halves agree on the row max through shared
//               memory and a 64-thread named barrier. O is rescaled in TMEM
//               only when the max grew by more than 2^8.
// Unlike the two-tile ping-pong of the narrower forward, the next scores'
// completion no longer implies that the previous P V product is done, so
// every P V product commits to pv_done. A rescale of O at tile j waits for
// P_{j-1} V's completion; its phase is unambiguous, since S_j was issued
// after P_{j-2} V (so that one is done) and P_j V is not issued before P_j
// is stored. The epilogue waits for the last product the same way.
// CTAs run head-major with the longest causal query tiles first; key tiles
// entirely above the causal diagonal are never loaded.
#include <type_traits>

#include "common.cuh"

namespace sdpa {
namespace {

struct Fwd256Layout {
  static constexpr int kQSlab = 128 * 128;   // 128 rows x 64 columns bf16
  static constexpr int kKVSlab = 64 * 128;   // 64 keys x 64 columns bf16
  static constexpr int kQBytes = 4 * kQSlab;    // 64 KB
  static constexpr int kKVBytes = 4 * kKVSlab;  // 32 KB per slot
  static constexpr int kSlots = 5;              // K / V ring
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kQBytes;
  // row-max / row-sum exchange between the two halves of a row: [half 2][row 128] fp32
  static constexpr int kRed = kKV + kSlots * kKVBytes;
  static constexpr int kBar = kRed + 2 * 128 * 4;
  // q_full, full[slots], empty[slots], s_full[2], p_full[2], pv_done
  static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align to 1024
  __host__ __device__ static constexpr uint32_t tmem_s(int b) { return 64u * b; }
  static constexpr uint32_t kTmemO = 256;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 320;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// Number of 64-key tiles that query rows [r0, r0+128) ∩ [0, Sq) can see.
__device__ __forceinline__ int kv64_tiles_for(int r0, int Sq, int Sk, bool causal) {
  if (r0 >= Sq || Sk <= 0) return 0;
  const int n = (Sk + 63) / 64;
  if (!causal) return n;
  return min(n, min(r0 + 127, Sq - 1) / 64 + 1);
}

struct Fwd256Item {
  int b, h, bh, q0, Sq, Sk, qs, ks, tb, n_kv;
  bool active;   // the tile holds query rows
  bool no_keys;  // a packed sequence with queries and no keys
};

// CTA x: query tile x of the head-major order, the longest causal tiles of a
// head first. p.n_q_tiles counts 128-row tiles here.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Fwd256Item fwd256_item(const FwdParams& p, int item) {
  Fwd256Item it;
  const int n_tiles = p.n_q_tiles;
  const int slot = item / n_tiles;
  int tile = item - slot * n_tiles;
  if (CAUSAL) tile = n_tiles - 1 - tile;
  it.b = slot / p.H;
  it.h = slot - it.b * p.H;
  it.bh = it.b * p.H + it.h;
  it.q0 = tile * 128;
  it.Sq = p.Sq;
  it.Sk = p.Sk;
  it.qs = 0;
  it.ks = 0;
  if (VARLEN) {
    it.qs = p.cu_q[it.b];
    it.Sq = p.cu_q[it.b + 1] - it.qs;
    it.ks = p.cu_k[it.b];
    it.Sk = p.cu_k[it.b + 1] - it.ks;
  }
  it.tb = VARLEN ? 0 : it.b;
  it.active = it.q0 < it.Sq;
  it.no_keys = it.active && it.Sk <= 0;
  it.n_kv = (it.active && !it.no_keys) ? kv64_tiles_for(it.q0, it.Sq, it.Sk, CAUSAL) : 0;
  return it;
}

template <bool CAUSAL, bool DROPOUT, bool VARLEN>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel_d256(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FwdParams p) {
  using L = Fwd256Layout;
  constexpr int NSL = L::kSlots;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;       // [slots]
  uint64_t* kv_empty = kv_full + NSL;  // [slots]
  uint64_t* s_full = kv_empty + NSL;  // [2]
  uint64_t* p_full = s_full + 2;   // [2]
  uint64_t* pv_done = p_full + 2;  // one phase per P V product
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Fwd256Item it = fwd256_item<CAUSAL, VARLEN>(p, blockIdx.x);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NSL; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 256);
    }
    mbar_init(pv_done, 1);
    *abort_word = 0u;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_holder, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl wc{abort_word, p.err, p.wait_limit_ns};
  const int n_kv = it.n_kv;
  // ring item n: K_{n/2} (n even) or V_{n/2} (n odd), in slot n % slots

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_kv > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(q_full, L::kQBytes);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        tma_load_4d(smem + L::kQ + s * L::kQSlab, &tm_q, q_full, s * 64, it.qs + it.q0, it.h,
                    it.tb);
      int n = 0;
      for (; n < 2 * n_kv; ++n) {
        const int sl = n % NSL;
        // a slot is free once the product reading its previous item is done
        if (n >= NSL) mbar_wait(&kv_empty[sl], ((n / NSL) - 1) & 1, wc, kSiteFwdKvEmpty);
        mbar_arrive_expect_tx(&kv_full[sl], L::kKVBytes);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          tma_load_4d(smem + L::kKV + sl * L::kKVBytes + s * L::kKVSlab, (n & 1) ? &tm_v : &tm_k,
                      &kv_full[sl], s * 64, it.ks + (n >> 1) * 64, it.h, it.tb);
        if (*abort_word) {
          ++n;
          break;
        }
      }
      if (*abort_word) {
        // give the loads still in flight time to land before the CTA exits
        mbar_wait_drain(q_full, 0, 2000000ull);
        for (int u = max(0, n - NSL); u < n; ++u)
          mbar_wait_drain(&kv_full[u % NSL], (u / NSL) & 1, 2000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one();
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t kIdO = idesc_bf16_f32(128, 256, false, true);
    const uint64_t qd = sdesc_sw128(sb + L::kQ, 16, 1024);
    auto issue_s = [&](int buf, int sl) {
      const uint64_t kd = sdesc_sw128(sb + L::kKV + sl * L::kKVBytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const uint32_t qoff = (kk >> 2) * L::kQSlab + (kk & 3) * 32;
        const uint32_t koff = (kk >> 2) * L::kKVSlab + (kk & 3) * 32;
        mma_bf16_ss_if(leader, tmem + L::tmem_s(buf), sdesc_add(qd, qoff), sdesc_add(kd, koff),
                       kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit_if(leader, &s_full[buf]);
      mma_commit_if(leader, &kv_empty[sl]);
    };
    auto issue_pv = [&](int buf, int sl, bool first) {
      // V is the MN-major B operand: 64-column slabs L::kKVSlab apart, 16 keys
      // (2048 bytes of 128-byte rows) per K step
      const uint64_t vd = sdesc_sw128(sb + L::kKV + sl * L::kKVBytes, L::kKVSlab, 1024);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_ts_if(leader, tmem + L::kTmemO, tmem + L::tmem_s(buf) + kk * 8,
                       sdesc_add(vd, kk * 2048), kIdO, (!first || kk > 0) ? 1u : 0u);
      mma_commit_if(leader, pv_done);
      mma_commit_if(leader, &kv_empty[sl]);
    };
    if (n_kv > 0) {
      mbar_wait(q_full, 0, wc, kSiteFwdQFull);
      mbar_wait(&kv_full[0], 0, wc, kSiteFwdKvFull);
      tc_fence_after();
      issue_s(0, 0);
      for (int j = 0; j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int nk = 2 * (j + 1);  // ring item of K_{j+1}
          mbar_wait(&kv_full[nk % NSL], (nk / NSL) & 1, wc, kSiteFwdKvFull);
          tc_fence_after();
          issue_s((j + 1) & 1, nk % NSL);
        }
        const int nv = 2 * j + 1;  // ring item of V_j
        mbar_wait(&p_full[j & 1], (j >> 1) & 1, wc, kSiteFwdPFull);
        mbar_wait(&kv_full[nv % NSL], (nv / NSL) & 1, wc, kSiteFwdKvFull);
        tc_fence_after();
        issue_pv(j & 1, nv % NSL, j == 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int half = warp >> 2;         // half of the tile's 64 keys
    const int row = threadIdx.x & 127;  // row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t pair_bar = 1 + (warp & 3);
    float* red = reinterpret_cast<float*>(smem + L::kRed);
    const float sl2 = p.scale_log2;
    const PhiloxKey pk = DROPOUT ? launch_key(p.pk, p.rng_dev) : p.pk;
    // the half's value v, shared with the partner half through the pair's one
    // slot: the first barrier makes sure the partner has read the previous
    // value, the second that it has written this one
    auto exchange = [&](float v) {
      named_barrier_sync(pair_bar, 64);
      red[half * 128 + row] = v;
      // also orders the partner's TMEM score reads before this warp's P
      // stores into the same columns
      tc_fence_before();
      named_barrier_sync(pair_bar, 64);
      tc_fence_after();
      return red[(1 - half) * 128 + row];
    };
    const int b = it.b, h = it.h, bh = it.bh, q0 = it.q0, Sq = it.Sq, Sk = it.Sk, qs = it.qs;
    const int qi = q0 + row;
    if (it.no_keys) {
      // no keys: the rows' outputs are 0 and their log-sum-exp is -inf
      if (half == 0 && qi < Sq) {
        uint16_t* o = static_cast<uint16_t*>(p.out_io.data) + h * p.out_io.sH +
                      static_cast<int64_t>(qs + qi) * p.out_io.sS;
        for (int c = 0; c < p.D_io; c += 8)
          *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
        p.lse[static_cast<size_t>(h) * p.total_q + qs + qi] = -INFINITY;
      }
    } else if (n_kv > 0) {
      const uint32_t tO = tmem + L::kTmemO + lane_base;
      float m = -INFINITY;  // running max of the raw scores of the row
      float l = 0.f;        // this half's running sum
      for (int j = 0; j < n_kv; ++j) {
        const int buf = j & 1;
        const uint32_t tS = tmem + L::tmem_s(buf) + lane_base;
        mbar_wait(&s_full[buf], (j >> 1) & 1, wc, kSiteFwdSFull);
        tc_fence_after();
        uint32_t r0[32];
        tmem_ld32(tS + 32 * half, r0);
        tmem_ld_wait(r0);
        float x[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(r0[c]);
        const int k0 = j * 64 + 32 * half;  // first key of this half
        if ((k0 + 32 > Sk) || (CAUSAL && k0 + 31 > q0)) {
          const int lim = CAUSAL ? min(Sk - k0, qi - k0 + 1) : (Sk - k0);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c >= lim) x[c] = -INFINITY;
        }
        float mp[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mp[u] = fmaxf(x[u], x[8 + u]);
#pragma unroll
        for (int u = 0; u < 8; ++u) mp[u] = fmax3(mp[u], x[16 + u], x[24 + u]);
        const float mh =
            fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], fmax3(mp[5], mp[6], mp[7])));
        const float m_new = fmaxf(m, fmaxf(mh, exchange(mh)));
        if (j == 0) {
          m = m_new;
        } else if (__any_sync(0xffffffffu, (m_new - m) * sl2 > 8.0f)) {
          // both halves of these rows take this branch (same rows, same
          // maxima). O must hold P_{j-1} V first: wait for that product.
          mbar_wait(pv_done, (j - 1) & 1, wc, kSiteFwdODone);
          tc_fence_after();
          const float alpha = ex2_approx((m - m_new) * sl2);
          l *= alpha;
          m = m_new;
#pragma unroll
          for (int c = 0; c < 4; ++c) {  // this half's 128 columns of O
            uint32_t o[32];
            tmem_ld32(tO + 128 * half + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + 128 * half + c * 32, o);
          }
        }
        const float neg = -m * sl2;

        // P = exp2(x*scale*log2e - m); with dropout P~ = keep ? P : 0, and the
        // 1/(1-p) is applied in the epilogue. The row sum takes P.
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk2[16];
        // mode 0: no dropout; 1, 3: the half row starts on a group boundary
        // (Sk a multiple of 4), so group g_row + t holds keys 4t .. 4t+3 and
        // is drawn where those keys are exponentiated (1: round keys from the
        // parameters, 3: the key read from device memory); 2: keep bits first
        auto exp_pack = [&](auto mode_c, uint64_t g_row, uint32_t keep) {
          constexpr int kMode = decltype(mode_c)::value;
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            float e[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) e[w] = ex2_approx(fmaf(x[c + w], sl2, neg));
            rs[(c >> 2) & 3] += (e[0] + e[1]) + (e[2] + e[3]);
            if constexpr (kMode == 1 || kMode == 3) {
              const uint4 u = kMode == 1
                                  ? philox_group_rk(g_row + (c >> 2), p.pk.off_lo, p.pk.off_hi, p.rk)
                                  : philox_group(g_row + (c >> 2), pk);
              const uint32_t thr = p.drop_threshold;
              e[0] = u.x >= thr ? e[0] : 0.f;
              e[1] = u.y >= thr ? e[1] : 0.f;
              e[2] = u.z >= thr ? e[2] : 0.f;
              e[3] = u.w >= thr ? e[3] : 0.f;
            } else if constexpr (kMode == 2) {
#pragma unroll
              for (int w = 0; w < 4; ++w) e[w] = ((keep >> (c + w)) & 1u) ? e[w] : 0.f;
            }
            pk2[c >> 1] = pack_bf16x2(e[0], e[1]);
            pk2[(c >> 1) + 1] = pack_bf16x2(e[2], e[3]);
          }
        };
        if (!DROPOUT) {
          exp_pack(std::integral_constant<int, 0>{}, 0, 0xffffffffu);
        } else {
          const uint64_t n0 = (counter_bh(b, h, p.b0, p.h0, p.H_total) * p.Sq_ctr + qi) *
                                  static_cast<uint64_t>(p.Sk_ctr) +
                              k0;
          if ((p.Sk_ctr & 3) == 0) {
            if (p.rng_dev == nullptr)
              exp_pack(std::integral_constant<int, 1>{}, n0 >> 2, 0u);
            else
              exp_pack(std::integral_constant<int, 3>{}, n0 >> 2, 0u);
          } else {
            uint32_t keep[1];
            keep_bits<1>(n0, p.drop_threshold, pk, keep);
            exp_pack(std::integral_constant<int, 2>{}, 0, keep[0]);
          }
        }
        // P (bf16 pairs) of keys [32h, 32h+32) -> S columns [16h, 16h+16);
        // they overwrite scores this warp pair has already read
        tmem_st16(tS + 16 * half, pk2);
        l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[buf]);
      }
      // ---------------------------------------------------------- epilogue
      const float l_row = l + exchange(l);
      mbar_wait(pv_done, (n_kv - 1) & 1, wc, kSiteFwdODone);
      tc_fence_after();
      const float inv_l = (DROPOUT ? p.drop_rescale : 1.f) / l_row;
      uint16_t* orow = static_cast<uint16_t*>(p.out_io.data) + it.tb * p.out_io.sB +
                       h * p.out_io.sH + static_cast<int64_t>(qs + qi) * p.out_io.sS;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // this half's 128 columns
        uint32_t o[32];
        tmem_ld32(tO + 128 * half + c * 32, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int col0 = 128 * half + c * 32 + q4 * 8;
          const uint32_t w0 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 1]) * inv_l);
          const uint32_t w1 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 3]) * inv_l);
          const uint32_t w2 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 5]) * inv_l);
          const uint32_t w3 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 7]) * inv_l);
          if (qi < Sq && col0 < p.D_io)
            *reinterpret_cast<uint4*>(orow + col0) = make_uint4(w0, w1, w2, w3);
        }
      }
      if (half == 0 && qi < Sq)
        p.lse[(VARLEN ? static_cast<size_t>(h) * p.total_q + qs : static_cast<size_t>(bh) * Sq) +
              qi] = m * (sl2 * kLn2) + __logf(l_row);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <bool C, bool DR, bool VL>
cudaError_t launch_fwd256_t(const CUtensorMap* maps, const FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_kernel_d256<C, DR, VL>;
  const int smem = Fwd256Layout::kAlloc;
  cudaError_t e = ensure_smem_attr<fwd_kernel_d256<C, DR, VL>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.n_q_tiles) * static_cast<unsigned>(p.B * p.H);
  kern<<<grid, Fwd256Layout::kThreads, smem, stream>>>(maps[0], maps[1], maps[2], p);
  return cudaGetLastError();
}

}  // namespace

// The forward for kernel head dim 256: one 128-row query tile per CTA
// (p.n_q_tiles = ceil(Sq / 128)); maps: q (box 64 x 128 rows), k and v
// (box 64 x 64 rows).
cudaError_t launch_fwd_d256(bool causal, bool dropout, const CUtensorMap* maps, const FwdParams& p,
                            cudaStream_t stream) {
  const bool varlen = p.cu_q != nullptr;
#define SDPA_FWD256_CASE(CC, RR)                                                  \
  if (causal == CC && dropout == RR)                                              \
    return varlen ? launch_fwd256_t<CC, RR, true>(maps, p, stream)                \
                  : launch_fwd256_t<CC, RR, false>(maps, p, stream);
  SDPA_FWD256_CASE(false, false)
  SDPA_FWD256_CASE(false, true)
  SDPA_FWD256_CASE(true, false)
  SDPA_FWD256_CASE(true, true)
#undef SDPA_FWD256_CASE
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
