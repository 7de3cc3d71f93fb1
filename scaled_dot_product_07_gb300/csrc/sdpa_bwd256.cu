// Main backward kernel for head dims 136..256 (kernel width 256; sdpfa_bwd
// of test_sdpa_loop_split, "DID loop split for SDPA", NVIDIA/Fuser PR 3711;
// probabilities recomputed from the stashed log-sum-exp, NVIDIA/Fuser issue
// 2278; dropout mask regenerated from the absolute index, "REDO of dropout
// support for mem eff #102038").
//
// At D = 256 the fp32 dK and dV of a 128-key tile would fill all 512 TMEM
// columns, so each 128-key tile of one (batch, head) is served by two CTAs,
// one per 128-column half of D: CTA half hd keeps dK[:, hd] and dV[:, hd]
// (128 columns each) and produces dQ[:, hd]. Both CTAs of a tile contract
// the full D for S^T = K Q^T and dP~^T = V dO^T (7/5 of the algorithmic
// flops). K is the A operand of S^T = K Q^T straight from TMEM (128 columns
// of bf16 pairs, stored there once by compute warpgroup A), so shared memory
// keeps only K[:, hd] (32 KB, for dQ) and V (64 KB), and the query steps are
// 32 rows (Q and dO 16 KB each per stage, 3 stages). 448 threads:
//   warp 13     TMA: K[:, hd], V once; Q_t, dO_t, lse2_t, Delta_t through the ring
//   warp 12     TMEM allocator and MMA issuer (converged warp, elected lane)
//   warps 0-3   compute warpgroup A (even steps), warps 4-7 B (odd steps):
//               thread = key row. P~^T (bf16) goes to TMEM as the A operand
//               of dV += P~^T dO[:, hd]; dS^T (bf16, 64-byte rows, 64-byte
//               swizzle) to shared memory as the operand of dK += dS^T
//               Q[:, hd] and dQ^T[hd] = K[:, hd]^T dS^T.
//   warps 8-11  dQ warpgroup: stages the step's dQ^T partial [32 rows x 128]
//               fp32 and reduces it into this half's rows of the fp32
//               accumulator (layout [B*H][2][Sq_pad][128]) with four bulk
//               reduce-adds.
// TMEM: dV [0,128), dK [128,256), two step buffers {S^T (32 columns),
// dP^T (32)} at 256 + 64 b, and K [384,512); a step's dQ^T partial (128 lanes = d, 32
// columns) overwrites its dP^T columns once the compute warpgroup has read
// them. MMA order per step t: S^T(t), dP^T(t), then dV, dK, dQ of step t-1.
#include "common.cuh"

namespace sdpa {
namespace {

struct B256 {
  static constexpr int kMq = 32;                  // query rows per step
  static constexpr int kStages = 3;               // Q / dO ring
  static constexpr int kKvSlab = 128 * 128;       // 128 keys x 64 columns bf16 (16 KB)
  static constexpr int kKvBytes = 4 * kKvSlab;    // 64 KB
  static constexpr int kQSlab = kMq * 128;        // 32 rows x 64 columns (4 KB)
  static constexpr int kQBytes = 4 * kQSlab;      // 16 KB
  static constexpr int kDsBytes = 128 * kMq * 2;  // [128 keys x 32 rows] bf16, 64-byte rows (8 KB)
  static constexpr int kDqBytes = kMq * 128 * 4;  // [32 rows x 128 d] fp32 staging (16 KB)
  static constexpr int kK = 0;                    // K[:, hd]: two slabs
  static constexpr int kV = kK + 2 * kKvSlab;
  static constexpr int kQ = kV + kKvBytes;
  static constexpr int kDO = kQ + kStages * kQBytes;
  static constexpr int kDs = kDO + kStages * kQBytes;  // [2]
  static constexpr int kDq = kDs + 2 * kDsBytes;
  static constexpr int kLse = kDq + kDqBytes;              // [kStages][32] fp32
  static constexpr int kDelta = kLse + kStages * kMq * 4;  // [kStages][32] fp32
  static constexpr int kBar = kDelta + kStages * kMq * 4;
  // kv_full, q_full[S], q_empty[S], and per step buffer b in {0,1}:
  // s_full, dp_full, p_full, ds_full, sp_empty, dq_full, dq_empty, ds_empty;
  // done, ktm_full (K stored in TMEM)
  static constexpr int kNumBars = 1 + 2 * kStages + 8 * 2 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemDV = 0, kTmemDK = 128, kTmemCols = 512;
  __host__ __device__ static constexpr uint32_t tmem_s(int b) { return 256u + 64u * b; }
  __host__ __device__ static constexpr uint32_t tmem_dp(int b) { return 288u + 64u * b; }
  static constexpr uint32_t kTmemK = 384;  // K as bf16 pairs, 128 columns
  static constexpr int kThreads = 448;
  static_assert(kAlloc <= 232448, "shared memory budget");
  static_assert(kDs % 1024 == 0, "dS^T tiles on swizzle-pattern boundaries");
};

template <bool CAUSAL, bool DROPOUT, bool VARLEN>
__global__ void __launch_bounds__(448, 1)
    bwd_main_kernel_d256(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk,
                         const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using L = B256;
  constexpr int NS = L::kStages;
  constexpr bool kInlineWaits = DROPOUT || VARLEN;
  constexpr int MQ = L::kMq;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + NS;
  uint64_t* s_full = q_empty + NS;  // each of these is [2], indexed by step buffer
  uint64_t* dp_full = s_full + 2;
  uint64_t* p_full = dp_full + 2;
  uint64_t* ds_full = p_full + 2;
  uint64_t* sp_empty = ds_full + 2;
  uint64_t* dq_full = sp_empty + 2;
  uint64_t* dq_empty = dq_full + 2;
  uint64_t* ds_empty = dq_empty + 2;
  uint64_t* done = ds_empty + 2;
  uint64_t* ktm_full = done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The two halves of a key tile are neighbouring CTAs (they read the same
  // K, V, Q and dO tiles from L2). Groups of kSlotGroup (batch, head) slots
  // in order; within a group key tile j of every slot before key tile j+1.
  constexpr int kSlotGroup = 8;
  const int hd = blockIdx.x & 1;
  const int cta = blockIdx.x >> 1;
  const int n_slots = p.B * p.H;
  const int per_group = kSlotGroup * p.n_kv_tiles;
  const int grp = cta / per_group;
  const int in_grp = cta - grp * per_group;
  const int grp_slots = min(kSlotGroup, n_slots - grp * kSlotGroup);
  const int kv_tile = in_grp / grp_slots;
  const int slot = grp * kSlotGroup + (in_grp - kv_tile * grp_slots);
  const int b = slot / p.H;
  const int h = slot - b * p.H;
  const int bh = b * p.H + h;
  const int k0 = kv_tile * 128;
  int Sq = p.Sq, Sk = p.Sk, qs = 0, ks = 0;
  if (VARLEN) {
    qs = p.cu_q[b];
    Sq = p.cu_q[b + 1] - qs;
    ks = p.cu_k[b];
    Sk = p.cu_k[b + 1] - ks;
    if (k0 >= Sk) return;  // no keys of the sequence in this tile
  }
  const int tb = VARLEN ? 0 : b;
  const int n_qt = (Sq + MQ - 1) / MQ;
  const int qt_first = CAUSAL ? min(k0 / MQ, n_qt) : 0;
  const int n_steps = n_qt - qt_first;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&dp_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&ds_full[x], 128);
      mbar_init(&sp_empty[x], 128);
      mbar_init(&dq_full[x], 1);
      mbar_init(&dq_empty[x], 128);
      mbar_init(&ds_empty[x], 1);
    }
    mbar_init(done, 1);
    mbar_init(ktm_full, 128);
    *abort_word = 0u;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(tmem_holder, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const WaitCtl wc{abort_word, p.err, p.wait_limit_ns};

  if (warp == 13) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_steps > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(kv_full, 6 * L::kKvSlab);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        tma_load_4d(smem + L::kV + s * L::kKvSlab, &tm_v, kv_full, s * 64, ks + k0, h, tb);
#pragma unroll
      for (int s = 0; s < 2; ++s)
        tma_load_4d(smem + L::kK + s * L::kKvSlab, &tm_k, kv_full, (2 * hd + s) * 64, ks + k0, h,
                    tb);
      int t = 0;
      for (; t < n_steps; ++t) {
        const int st = t % NS;
        const int i0 = (qt_first + t) * MQ;
        if (t >= NS) mbar_wait_t<kInlineWaits>(&q_empty[st], ((t / NS) - 1) & 1, wc, kSiteBwdQEmpty);
        mbar_arrive_expect_tx(&q_full[st], 2 * L::kQBytes + 2 * MQ * 4);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          tma_load_4d(smem + L::kQ + st * L::kQBytes + s * L::kQSlab, &tm_q, &q_full[st], s * 64,
                      qs + i0, h, tb);
          tma_load_4d(smem + L::kDO + st * L::kQBytes + s * L::kQSlab, &tm_do, &q_full[st],
                      s * 64, qs + i0, h, tb);
        }
        const size_t vec = static_cast<size_t>(bh) * p.Sq_pad + i0;
        bulk_load(smem + L::kLse + st * MQ * 4, p.lse2 + vec, MQ * 4, &q_full[st]);
        bulk_load(smem + L::kDelta + st * MQ * 4, p.delta + vec, MQ * 4, &q_full[st]);
        if (*abort_word) {
          ++t;
          break;
        }
      }
      if (*abort_word) {
        mbar_wait_drain(kv_full, 0, 2000000ull);
        for (int u = max(0, t - NS); u < t; ++u)
          mbar_wait_drain(&q_full[u % NS], (u / NS) & 1, 2000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 12) {
    // ------------------------------------------------------------ MMA issuer
    if (n_steps > 0) {
      const uint32_t leader = elect_one();
      constexpr uint32_t kIdSP = idesc_bf16_f32(128, MQ, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_bf16_f32(128, 128, false, true);  // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, MQ, true, true);     // dQ^T
      const uint64_t kd_v = sdesc_sw128(sb + L::kV, 16, 1024);  // V, K-major
      // K[:, hd] as the MN-major A operand of dQ^T (M = 128 d in two 64-column
      // slabs, K = keys)
      const uint64_t kd_kmn = sdesc_sw128(sb + L::kK, L::kKvSlab, 1024);
      auto finish_step = [&](int u) {
        const int x = u & 1;
        const int st = u % NS;
        // Q[:, hd], dO[:, hd] as MN-major B operands (N = 128 d, K = rows)
        const uint64_t d_qmn =
            sdesc_sw128(sb + L::kQ + st * L::kQBytes + hd * 2 * L::kQSlab, L::kQSlab, 1024);
        const uint64_t d_omn =
            sdesc_sw128(sb + L::kDO + st * L::kQBytes + hd * 2 * L::kQSlab, L::kQSlab, 1024);
        // dS^T [128 keys x 32 rows], 64-byte rows: K-major A of dK, MN-major B of dQ^T
        const uint64_t d_ds = sdesc_sw64(sb + L::kDs + x * L::kDsBytes, 16, 512);
        const uint64_t d_dsmn = sdesc_sw64(sb + L::kDs + x * L::kDsBytes, L::kDsBytes, 512);
        mbar_wait_t<kInlineWaits>(&p_full[x], (u >> 1) & 1, wc, kSiteBwdPFull);
        tc_fence_after();
        // dV[:, hd] += P~^T dO[:, hd]: A = P~^T bf16 in TMEM (16 columns)
#pragma unroll
        for (int kk = 0; kk < MQ / 16; ++kk)
          mma_bf16_ts_if(leader, tmem + L::kTmemDV, tmem + L::tmem_s(x) + kk * 8,
                         sdesc_add(d_omn, kk * 2048), kIdKV, (u > 0 || kk > 0) ? 1u : 0u);
        mbar_wait_t<kInlineWaits>(&ds_full[x], (u >> 1) & 1, wc, kSiteBwdDsFull);
        tc_fence_after();
        // dK[:, hd] += dS^T Q[:, hd]
#pragma unroll
        for (int kk = 0; kk < MQ / 16; ++kk)
          mma_bf16_ss_if(leader, tmem + L::kTmemDK, sdesc_add(d_ds, kk * 32),
                         sdesc_add(d_qmn, kk * 2048), kIdKV, (u > 0 || kk > 0) ? 1u : 0u);
        // dQ^T[hd] [128 x MQ] = K[:, hd]^T dS^T into this step's dP^T columns
        // (read by the compute warpgroup before it signalled ds_full)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ss_if(leader, tmem + L::tmem_dp(x), sdesc_add(kd_kmn, kk * 2048),
                         sdesc_add(d_dsmn, kk * 1024), kIdQ, kk > 0 ? 1u : 0u);
        mma_commit_if(leader, &dq_full[x]);
        mma_commit_if(leader, &q_empty[st]);
        mma_commit_if(leader, &ds_empty[x]);
      };
      mbar_wait_t<kInlineWaits>(kv_full, 0, wc, kSiteBwdKvFull);
      mbar_wait_t<kInlineWaits>(ktm_full, 0, wc, kSiteBwdKvFull);
      tc_fence_after();
      for (int t = 0; t < n_steps; ++t) {
        const int x = t & 1;
        const int st = t % NS;
        const uint64_t d_q = sdesc_sw128(sb + L::kQ + st * L::kQBytes, 16, 1024);
        const uint64_t d_o = sdesc_sw128(sb + L::kDO + st * L::kQBytes, 16, 1024);
        mbar_wait_t<kInlineWaits>(&q_full[st], (t / NS) & 1, wc, kSiteBwdQFull);
        if (t >= 2) mbar_wait_t<kInlineWaits>(&sp_empty[x], ((t >> 1) - 1) & 1, wc, kSiteBwdSpEmpty);
        tc_fence_after();
        // S^T = K Q^T (M = 128 keys, N = 32 rows, K = 256 d): K from TMEM, 16
        // d (8 columns) per product
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint32_t qoff = (kk >> 2) * L::kQSlab + (kk & 3) * 32;
          mma_bf16_ts_if(leader, tmem + L::tmem_s(x), tmem + L::kTmemK + kk * 8,
                         sdesc_add(d_q, qoff), kIdSP, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(leader, &s_full[x]);
        // the dP^T columns held dQ^T(t-2) until the dQ warpgroup read it out
        if (t >= 2) {
          mbar_wait_t<kInlineWaits>(&dq_empty[x], ((t >> 1) - 1) & 1, wc, kSiteBwdDqEmpty);
          tc_fence_after();
        }
        // dP~^T = V dO^T
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kKvSlab + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * L::kQSlab + (kk & 3) * 32;
          mma_bf16_ss_if(leader, tmem + L::tmem_dp(x), sdesc_add(kd_v, koff), sdesc_add(d_o, qoff),
                         kIdSP, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(leader, &dp_full[x]);
        if (t >= 1) finish_step(t - 1);
      }
      finish_step(n_steps - 1);
      mma_commit_if(leader, done);
      mbar_wait_drain(done, 0, 2000000000ull);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute warpgroups A, B
    const int x = warp >> 2;  // step parity handled by this warpgroup
    const int r = threadIdx.x & 127;
    const int kj = k0 + r;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + L::tmem_s(x) + lane_base;
    const uint32_t tDP = tmem + L::tmem_dp(x) + lane_base;
    const uint32_t da = sb + L::kDs + x * L::kDsBytes;
    const PhiloxKey pk = DROPOUT ? launch_key(p.pk, p.rng_dev) : p.pk;
    if (x == 0 && n_steps > 0) {
      // K row kj (all 256 columns) into TMEM lane r as bf16 pairs: column c
      // holds elements 2c, 2c+1 (zeros past Sk and past the caller's D)
      const uint16_t* krow = static_cast<const uint16_t*>(p.k_io.data) + tb * p.k_io.sB +
                             h * p.k_io.sH + static_cast<int64_t>(ks + kj) * p.k_io.sS;
      const uint32_t tK = tmem + L::kTmemK + lane_base;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {  // 64 elements, 32 columns, at a time
        uint32_t w[32];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const int e0 = cc * 64 + q8 * 8;
          uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
          if (kj < Sk && e0 < p.D_io) v4 = *reinterpret_cast<const uint4*>(krow + e0);
          w[4 * q8 + 0] = v4.x;
          w[4 * q8 + 1] = v4.y;
          w[4 * q8 + 2] = v4.z;
          w[4 * q8 + 3] = v4.w;
        }
        tmem_st32(tK + cc * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ktm_full);
    }
    for (int t = x, k = 0; t < n_steps; t += 2, ++k) {
      const int st = t % NS;
      const int i0 = (qt_first + t) * MQ;
      const uint32_t lse_s = sb + L::kLse + st * MQ * 4;
      const uint32_t del_s = sb + L::kDelta + st * MQ * 4;
      // keep bits of the step's 32 rows of this key: drawn while the tensor
      // core computes S^T
      uint32_t kb = 0xffffffffu;
      if (DROPOUT) {
        const uint64_t n_base = (counter_bh(b, h, p.b0, p.h0, p.H_total) * p.Sq_ctr + i0) *
                                    static_cast<uint64_t>(p.Sk_ctr) +
                                kj;
        if ((p.Sk_ctr & 3) == 0) {
          uint32_t kb1[1];
          keep_bits_quad<1>(n_base, static_cast<uint64_t>(p.Sk_ctr), p.drop_threshold, pk, kb1);
          kb = kb1[0];
        } else {
#pragma unroll
          for (int c = 0; c < MQ; ++c) {
            const bool kp =
                keep_one(n_base + static_cast<uint64_t>(c) * p.Sk_ctr, p.drop_threshold, pk);
            if (!kp) kb &= ~(1u << c);
          }
        }
      }
      mbar_wait_t<kInlineWaits>(&q_full[st], (t / NS) & 1, wc, kSiteBwdQFull);
      mbar_wait_t<kInlineWaits>(&s_full[x], k & 1, wc, kSiteBwdSFull);
      tc_fence_after();
      float pv[MQ];
      {
        uint32_t r0[32];
        tmem_ld32(tS, r0);
        tmem_ld_wait(r0);
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c] = __uint_as_float(r0[c]);
      }
      const bool need_mask = (k0 + 128 > Sk) || (CAUSAL && i0 < k0 + 127);
      const int first_vis = kj >= Sk ? (1 << 30) : (CAUSAL ? kj - i0 : 0);
#pragma unroll
      for (int c = 0; c < MQ; ++c) {
        float e = ex2_approx(fmaf(pv[c], p.scale_log2, -ld_shared_f32(lse_s + c * 4)));
        if (need_mask && c < first_vis) e = 0.f;
        pv[c] = e;
      }
      {
        // P~^T (bf16) into this step's S^T columns [0, 16) of TMEM
        uint32_t pk16[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int e = 2 * c;
          float a = pv[e], bb = pv[e + 1];
          if (DROPOUT) {
            a = ((kb >> e) & 1u) ? a * p.drop_rescale : 0.f;
            bb = ((kb >> (e + 1)) & 1u) ? bb * p.drop_rescale : 0.f;
          }
          pk16[c] = pack_bf16x2(a, bb);
        }
        tmem_st16(tS, pk16);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&p_full[x]);

      mbar_wait_t<kInlineWaits>(&dp_full[x], k & 1, wc, kSiteBwdDpFull);
      tc_fence_after();
      if (k >= 1) mbar_wait_t<kInlineWaits>(&ds_empty[x], (k - 1) & 1, wc, kSiteBwdPdsEmpty);
      {
        uint32_t d[32];
        tmem_ld32(tDP, d);
        tmem_ld_wait(d);
        float ds[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float g = __uint_as_float(d[i]);
          if (DROPOUT) g = ((kb >> i) & 1u) ? g * p.drop_rescale : 0.f;
          ds[i] = pv[i] * (g - ld_shared_f32(del_s + i * 4));
        }
        // row r of dS^T: 64 bytes, four 16-byte chunks in the 64-byte swizzle
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(da + sw64_offset(r, c), pack_bf16x2(ds[8 * c + 0], ds[8 * c + 1]),
                       pack_bf16x2(ds[8 * c + 2], ds[8 * c + 3]),
                       pack_bf16x2(ds[8 * c + 4], ds[8 * c + 5]),
                       pack_bf16x2(ds[8 * c + 6], ds[8 * c + 7]));
      }
      tc_fence_before();
      mbar_arrive(&sp_empty[x]);
      fence_async_smem();
      mbar_arrive(&ds_full[x]);
    }
  } else {
    // ------------------------------------------------------------ dQ warpgroup (warps 8-11)
    const int lt = threadIdx.x - 256;  // TMEM lane = column of this half
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t qa = sb + L::kDq;
    float* part = p.dq_part ? p.dq_part + static_cast<size_t>(kv_tile) * p.part_stride : nullptr;
    for (int t = 0; t < n_steps; ++t) {
      const int x = t & 1;
      const int i0 = (qt_first + t) * MQ;
      mbar_wait_t<kInlineWaits>(&dq_full[x], (t >> 1) & 1, wc, kSiteBwdDqFull);
      tc_fence_after();
      uint32_t r0[32];
      tmem_ld32(tmem + L::tmem_dp(x) + lane_base, r0);
      tmem_ld_wait(r0);
      tc_fence_before();
      mbar_arrive(&dq_empty[x]);
      // [MQ rows][128] fp32; each warp's first lane reduces (deterministic
      // mode: stores) eight rows, 4 KB
      if ((lt & 31) == 0) bulk_wait_read_all();  // the previous copies have read the tile
      named_barrier_sync(2, 128);
#pragma unroll
      for (int c = 0; c < 32; ++c) st_shared_f32(qa + (c * 128 + lt) * 4, __uint_as_float(r0[c]));
      fence_async_smem();
      named_barrier_sync(2, 128);
      if ((lt & 31) == 0) {
        const int hh = lt >> 5;
        dq_out(p.dq_acc, part,
               ((static_cast<size_t>(bh) * 2 + hd) * p.Sq_pad + i0 + 8 * hh) * 128,
               smem + L::kDq + hh * (L::kDqBytes / 4), L::kDqBytes / 4);
        bulk_commit();
      }
    }
    if ((lt & 31) == 0) bulk_wait_all();
  }

  // ------------------------------------------------------------ epilogue: dV (A), dK (B)
  if (warp < 8) {
    const bool is_dv = warp < 4;
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t acc = tmem + (is_dv ? L::kTmemDV : L::kTmemDK) + lane_base;
    const uint32_t stage = sb + (is_dv ? L::kK : L::kV);  // K/V tiles are dead after `done`
    const float mul = is_dv ? 1.f : p.scale;
    const bool direct = VARLEN && (k0 + 128 > Sk);
    if (n_steps > 0) {
      mbar_wait_t<kInlineWaits>(done, 0, wc, kSiteBwdDone);
      tc_fence_after();
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
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
        const int col0 = c * 32 + q4 * 8;  // column within this half
        const uint32_t w0 = pack_bf16x2(v[q4 * 8 + 0], v[q4 * 8 + 1]);
        const uint32_t w1 = pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]);
        const uint32_t w2 = pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]);
        const uint32_t w3 = pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]);
        if (direct) {
          if (k0 + r < Sk && 128 * hd + col0 < p.D_io) {
            const StridedBf16& o = is_dv ? p.dv_io : p.dk_io;
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(o.data) + h * o.sH +
                                      static_cast<int64_t>(ks + k0 + r) * o.sS + 128 * hd +
                                      col0) = make_uint4(w0, w1, w2, w3);
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
        for (int s = 0; s < 2; ++s)  // column slabs of this half the caller's head dim reaches
          if (128 * hd + s * 64 < p.D_io)
            tma_store_4d(is_dv ? &tm_dv : &tm_dk, smem + (is_dv ? L::kK : L::kV) + s * L::kKvSlab,
                         128 * hd + s * 64, ks + k0, h, tb);
        bulk_commit();
        bulk_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <bool C, bool DR, bool VL>
cudaError_t launch256_t(const CUtensorMap* m, const BwdParams& p, cudaStream_t stream) {
  auto kern = bwd_main_kernel_d256<C, DR, VL>;
  const int smem = B256::kAlloc;
  cudaError_t e = ensure_smem_attr<bwd_main_kernel_d256<C, DR, VL>>(smem);
  if (e != cudaSuccess) return e;
  // two CTAs (column halves) per 128-key tile of every (batch, head)
  const unsigned grid =
      2u * static_cast<unsigned>(p.n_kv_tiles) * static_cast<unsigned>(p.B * p.H);
  kern<<<grid, B256::kThreads, smem, stream>>>(m[0], m[1], m[2], m[3], m[4], m[5], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_d256(bool causal, bool dropout, const CUtensorMap* maps,
                                 const BwdParams& p, cudaStream_t stream) {
  const bool varlen = p.cu_q != nullptr;
#define SDPA_BWD256_CASE(CC, RR)                                                 \
  if (causal == CC && dropout == RR)                                             \
    return varlen ? launch256_t<CC, RR, true>(maps, p, stream)                   \
                  : launch256_t<CC, RR, false>(maps, p, stream);
  SDPA_BWD256_CASE(false, false)
  SDPA_BWD256_CASE(false, true)
  SDPA_BWD256_CASE(true, false)
  SDPA_BWD256_CASE(true, true)
#undef SDPA_BWD256_CASE
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
