// Main backward kernel for head dim 128 (sdpfa_bwd of test_sdpa_loop_split,
// "DID loop split for SDPA", NVIDIA/Fuser PR 3711; probabilities recomputed
// from the stashed log-sum-exp, NVIDIA/Fuser issue 2278; dropout mask
// regenerated from the absolute index, "REDO of dropout support for mem eff
// #102038").
//
// One CTA per 128-key tile of one (batch, head); it walks the 64-row query
// steps that can see its keys. 448 threads:
//   warp 13     TMA: K, V once; Q_t, dO_t, lse2_t, Delta_t through a 3-stage ring
//   warp 12     TMEM allocator and MMA issuer (the warp runs converged; one
//               elected lane issues the tcgen05 instructions)
//   warps 0-3   compute warpgroup A (even steps), warps 4-7 B (odd steps):
//               thread = key row. P^T = exp2(S^T*scale*log2e - lse2) (masked,
//               dropout applied) is stored as bf16 into TMEM (A operand of
//               dV += P~^T dO); dS^T = P^T (dP~^T keep/(1-p) - Delta) is
//               stored as bf16 into shared memory (B operand of dQ^T) and
//               into the step's S^T columns [32, 64) of TMEM (A operand of
//               dK += dS^T Q, which so reads only Q from shared memory: the
//               kernel is bound by shared-memory bandwidth).
//   warps 8-11  dQ warpgroup: reads the dQ^T partial of a step from TMEM,
//               stages it fp32 [64 x 128] and reduces it into the global fp32
//               accumulator with four bulk reduce-adds (one per warp).
// TMEM (512 columns): dV [0,128), dK [128,256), and two step buffers
// {S^T, dP^T} at [256,384) and [384,512). A step's dQ^T partial (M = D =
// 128 lanes, 64 columns) overwrites its own dP^T columns, which the compute
// warpgroup has read before it hands over dS^T; the next S^T into the
// buffer therefore waits only for the compute warpgroup, and the next dP^T
// for the dQ readout.
// MMA order per step t: S^T(t), dP^T(t), then dV, dK, dQ of step t-1, so
// the tensor core computes the next step's products while a compute
// warpgroup works on the current one.
#include <type_traits>

#include "common.cuh"

namespace sdpa {
namespace {

// With an attention bias, the Q / dO ring has 2 stages instead of 3 and the
// freed 32 KB hold the step's bias tile [64 query rows x 128 keys] (bf16,
// unswizzled), loaded by TMA with Q and dO.
template <bool BIAS>
struct B128 {
  static constexpr int D = 128;
  static constexpr int kMq = 64;                 // query rows per step
  static constexpr int kStages = BIAS ? 2 : 3;   // Q / dO ring
  static constexpr int kKvSlab = 128 * 128;      // 128 rows x 128 bytes
  static constexpr int kKvBytes = 128 * D * 2;   // 32 KB
  static constexpr int kQSlab = kMq * 128;       // 8 KB
  static constexpr int kQBytes = kMq * D * 2;    // 16 KB
  static constexpr int kDsBytes = 128 * kMq * 2; // [128 keys x 64 q] bf16 = 16 KB
  static constexpr int kDqBytes = kMq * D * 4;   // 32 KB fp32 staging
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKvBytes;
  static constexpr int kQ = kV + kKvBytes;
  static constexpr int kDO = kQ + kStages * kQBytes;
  static constexpr int kDs = kDO + kStages * kQBytes;        // [2]
  static constexpr int kDq = kDs + 2 * kDsBytes;
  static constexpr int kLse = kDq + kDqBytes;                // [kStages][64] fp32
  static constexpr int kDelta = kLse + kStages * kMq * 4;    // [kStages][64] fp32
  static constexpr int kBiasBytes = kMq * 128 * 2;            // 16 KB
  static constexpr int kBiasT = BIAS ? (kDelta + kStages * kMq * 4 + 1023) / 1024 * 1024
                                     : kDelta + kStages * kMq * 4;  // [kStages] tiles
  static constexpr int kBar = kBiasT + (BIAS ? kStages * kBiasBytes : 0);
  // kv_full, q_full[S], q_empty[S], and per step buffer b in {0,1}:
  // s_full, dp_full, p_full, ds_full, sp_empty, dq_full, dq_empty, ds_empty; done
  // (bias: + dbias_read[S], the dbias tile's TMA store has read its stage)
  static constexpr int kNumBars = 1 + 2 * kStages + 8 * 2 + 1 + (BIAS ? kStages : 0);
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemDV = 0, kTmemDK = 128, kTmemCols = 512;
  __host__ __device__ static constexpr uint32_t tmem_s(int b) { return 256u + 128u * b; }
  __host__ __device__ static constexpr uint32_t tmem_dp(int b) { return 320u + 128u * b; }
  static constexpr int kThreads = 448;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

__device__ __forceinline__ void touch32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31]));
}

template <bool CAUSAL, bool DROPOUT, bool BIAS, bool VARLEN>
__global__ void __launch_bounds__(448, 1)
    bwd_main_kernel_d128(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk,
                         const __grid_constant__ CUtensorMap tm_dv,
                         const __grid_constant__ CUtensorMap tm_bias,
                         const __grid_constant__ CUtensorMap tm_dbias,
                         const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using L = B128<BIAS>;
  constexpr int NS = L::kStages;
  // waits poll inline in the variants whose compute loops are short of
  // registers (dropout, bias, packed batches: spills around the call of an
  // out-of-line poll); the plain variants keep the smaller out-of-line form
  constexpr bool kInlineWaits = DROPOUT || BIAS || VARLEN;
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
  uint64_t* dbias_read = done + 1;  // [NS], bias only
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Groups of kSlotGroup (batch, head) slots in order (a group's Q and dO
  // stay in L2 while its key tiles run); within a group key tile j of every
  // slot before key tile j+1, so the low key tiles, which see the most
  // causal query rows, go first and the grid ends on short ones.
  constexpr int kSlotGroup = 8;
  const int n_slots = p.B * p.H;
  const int per_group = kSlotGroup * p.n_kv_tiles;
  const int grp = blockIdx.x / per_group;
  const int in_grp = blockIdx.x - grp * per_group;
  const int grp_slots = min(kSlotGroup, n_slots - grp * kSlotGroup);
  const int kv_tile = in_grp / grp_slots;
  const int slot = grp * kSlotGroup + (in_grp - kv_tile * grp_slots);
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
    if (BIAS)
      for (int s = 0; s < NS; ++s) mbar_init(&dbias_read[s], 1);
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
      mbar_arrive_expect_tx(kv_full, 2 * L::kKvBytes);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        tma_load_4d(smem + L::kK + s * L::kKvSlab, &tm_k, kv_full, s * 64, ks + k0, h, tb);
        tma_load_4d(smem + L::kV + s * L::kKvSlab, &tm_v, kv_full, s * 64, ks + k0, h, tb);
      }
      for (int t = 0; t < n_steps; ++t) {
        const int st = t % NS;
        const int i0 = (qt_first + t) * MQ;
        if (t >= NS) mbar_wait_t<kInlineWaits>(&q_empty[st], ((t / NS) - 1) & 1, wc, kSiteBwdQEmpty);
        // the bias stage also held step t-NS's dbias tile until its store read it
        if (BIAS && p.dbias.data != nullptr && t >= NS)
          mbar_wait_t<kInlineWaits>(&dbias_read[st], ((t / NS) - 1) & 1, wc, kSiteBwdQEmpty);
        mbar_arrive_expect_tx(&q_full[st],
                              2 * L::kQBytes + 2 * MQ * 4 + (BIAS ? L::kBiasBytes : 0));
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          tma_load_4d(smem + L::kQ + st * L::kQBytes + s * L::kQSlab, &tm_q, &q_full[st], s * 64,
                      qs + i0, h, tb);
          tma_load_4d(smem + L::kDO + st * L::kQBytes + s * L::kQSlab, &tm_do, &q_full[st],
                      s * 64, qs + i0, h, tb);
        }
        const size_t vec = static_cast<size_t>(bh) * p.Sq_pad + i0;
        bulk_load(smem + L::kLse + st * MQ * 4, p.lse2 + vec, MQ * 4, &q_full[st]);
        bulk_load(smem + L::kDelta + st * MQ * 4, p.delta + vec, MQ * 4, &q_full[st]);
        if (BIAS)  // rows past Sq and keys past Sk read as zeros
          tma_load_4d(smem + L::kBiasT + st * L::kBiasBytes, &tm_bias, &q_full[st], k0, i0,
                      p.bias.sH == 0 ? 0 : h, p.bias.sB == 0 ? 0 : b);
      }
      if (*abort_word) {
        for (int t = max(0, n_steps - NS); t < n_steps; ++t)
          mbar_wait_drain(&q_full[t % NS], (t / NS) & 1, 2000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 12) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and descriptor arithmetic are
    // warp-uniform); one elected lane issues the tcgen05 instructions.
    if (n_steps > 0) {
      const uint32_t leader = elect_one();
      constexpr uint32_t kIdSP = idesc_bf16_f32(128, MQ, false, false);  // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_bf16_f32(128, 128, false, true);  // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, MQ, true, true);     // dQ^T
      // descriptor bases; per-MMA steps add compile-time offsets
      const uint64_t kd_k = sdesc_sw128(sb + L::kK, 16, 1024);          // K, K-major
      const uint64_t kd_v = sdesc_sw128(sb + L::kV, 16, 1024);          // V, K-major
      const uint64_t kd_kmn = sdesc_sw128(sb + L::kK, L::kKvSlab, 1024);  // K as MN-major A
      // dV, dK and dQ of step u (buffer u & 1, stage u % NS)
      auto finish_step = [&](int u) {
        const int x = u & 1;
        const int st = u % NS;
        const uint64_t d_qmn = sdesc_sw128(sb + L::kQ + st * L::kQBytes, L::kQSlab, 1024);
        const uint64_t d_omn = sdesc_sw128(sb + L::kDO + st * L::kQBytes, L::kQSlab, 1024);
        const uint64_t d_dsmn = sdesc_sw128(sb + L::kDs + x * L::kDsBytes, L::kDsBytes, 1024);
        mbar_wait_t<kInlineWaits>(&p_full[x], (u >> 1) & 1, wc, kSiteBwdPFull);
        tc_fence_after();
        // dV += P~^T dO: A = P~^T bf16 in TMEM (32 columns), B = dO MN-major
#pragma unroll
        for (int kk = 0; kk < MQ / 16; ++kk)
          mma_bf16_ts_if(leader, tmem + L::kTmemDV, tmem + L::tmem_s(x) + kk * 8,
                         sdesc_add(d_omn, kk * 2048), kIdKV, (u > 0 || kk > 0) ? 1u : 0u);
        mbar_wait_t<kInlineWaits>(&ds_full[x], (u >> 1) & 1, wc, kSiteBwdDsFull);
        tc_fence_after();
        // dK += dS^T Q: A = dS^T bf16 in TMEM (S^T columns [32, 64), written by
        // the compute warpgroup beside its shared-memory copy), B = Q MN-major
#pragma unroll
        for (int kk = 0; kk < MQ / 16; ++kk)
          mma_bf16_ts_if(leader, tmem + L::kTmemDK, tmem + L::tmem_s(x) + 32 + kk * 8,
                         sdesc_add(d_qmn, kk * 2048), kIdKV, (u > 0 || kk > 0) ? 1u : 0u);
        // dQ^T [D x MQ] = K^T dS^T: A = K tile MN-major, B = dS^T MN-major; it
        // overwrites this step's dP^T columns (the compute warpgroup read them
        // before it signalled ds_full), so that the next S^T into this buffer
        // need not wait for the dQ^T readout
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ss_if(leader, tmem + L::tmem_dp(x), sdesc_add(kd_kmn, kk * 2048),
                         sdesc_add(d_dsmn, kk * 2048), kIdQ, kk > 0 ? 1u : 0u);
        mma_commit_if(leader, &dq_full[x]);
        mma_commit_if(leader, &q_empty[st]);
        mma_commit_if(leader, &ds_empty[x]);
      };
      mbar_wait_t<kInlineWaits>(kv_full, 0, wc, kSiteBwdKvFull);
      for (int t = 0; t < n_steps; ++t) {
        const int x = t & 1;
        const int st = t % NS;
        const uint64_t d_q = sdesc_sw128(sb + L::kQ + st * L::kQBytes, 16, 1024);
        const uint64_t d_o = sdesc_sw128(sb + L::kDO + st * L::kQBytes, 16, 1024);
        mbar_wait_t<kInlineWaits>(&q_full[st], (t / NS) & 1, wc, kSiteBwdQFull);
        // step buffer x: S^T(t-2) and dP^T(t-2) read by the compute warpgroup
        if (t >= 2) mbar_wait_t<kInlineWaits>(&sp_empty[x], ((t >> 1) - 1) & 1, wc, kSiteBwdSpEmpty);
        tc_fence_after();
        // S^T = K Q^T and dP~^T = V dO^T  (M = 128 keys, N = MQ, K = D)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kKvSlab + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * L::kQSlab + (kk & 3) * 32;
          mma_bf16_ss_if(leader, tmem + L::tmem_s(x), sdesc_add(kd_k, koff), sdesc_add(d_q, qoff),
                         kIdSP, kk > 0 ? 1u : 0u);
        }
        mma_commit_if(leader, &s_full[x]);
        // the dP^T columns held dQ^T(t-2) until the dQ warpgroup read it out
        if (t >= 2) {
          mbar_wait_t<kInlineWaits>(&dq_empty[x], ((t >> 1) - 1) & 1, wc, kSiteBwdDqEmpty);
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
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
    for (int t = x, k = 0; t < n_steps; t += 2, ++k) {
      const int st = t % NS;
      const int i0 = (qt_first + t) * MQ;
      const uint32_t lse_s = sb + L::kLse + st * MQ * 4;
      const uint32_t del_s = sb + L::kDelta + st * MQ * 4;
      // this step's bias tile [MQ query rows x 128 keys] (bf16, row-major),
      // loaded with Q and dO: column r is this thread's key
      const uint32_t bias_s = sb + L::kBiasT + st * L::kBiasBytes + 2 * r;
      // the step's dropout keep bits depend only on the indices: drawn while
      // the tensor core computes S^T
      uint32_t kb[2] = {0xffffffffu, 0xffffffffu};
      // with the forward's stored bits: lane l reads rows i0 + l and i0 + 32 + l
      // of its warp's 32 keys (transposed to one word per key after the waits)
      const bool stored = DROPOUT && !BIAS && !VARLEN && p.drop_bits != nullptr;
      uint32_t sw[2] = {0u, 0u};
      if (stored) {
        const uint32_t* wp =
            p.drop_bits + (static_cast<size_t>(bh) * p.bits_kw + (k0 >> 5) + (warp & 3)) * p.bits_rows +
            i0 + lane;
        sw[0] = wp[0];
        sw[1] = wp[32];
      } else if (DROPOUT) {
        const uint64_t n_base = (counter_bh(b, h, p.b0, p.h0, p.H_total) * p.Sq_ctr + i0) *
                                    static_cast<uint64_t>(p.Sk_ctr) +
                                kj;
        if ((p.Sk_ctr & 3) == 0) {
          keep_bits_quad<2>(n_base, static_cast<uint64_t>(p.Sk_ctr), p.drop_threshold, pk, kb);
        } else {
#pragma unroll
          for (int c = 0; c < MQ; ++c) {
            const bool kp =
                keep_one(n_base + static_cast<uint64_t>(c) * p.Sk_ctr, p.drop_threshold, pk);
            if (!kp) kb[c >> 5] &= ~(1u << (c & 31));
          }
        }
      }
      mbar_wait_t<kInlineWaits>(&q_full[st], (t / NS) & 1, wc, kSiteBwdQFull);
      mbar_wait_t<kInlineWaits>(&s_full[x], k & 1, wc, kSiteBwdSFull);
      tc_fence_after();
      if (stored) {
        kb[0] = warp_transpose32(sw[0], lane);
        kb[1] = warp_transpose32(sw[1], lane);
      }
      float pv[MQ];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tS, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld_wait(r0);
        touch32(r1);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          pv[c] = __uint_as_float(r0[c]);
          pv[32 + c] = __uint_as_float(r1[c]);
        }
      }
      const bool need_mask = (k0 + 128 > Sk) || (CAUSAL && i0 < k0 + 127);
      const int first_vis = kj >= Sk ? (1 << 30) : (CAUSAL ? kj - i0 : 0);
#pragma unroll
      for (int c = 0; c < MQ; ++c) {
        float arg = fmaf(pv[c], p.scale_log2, -ld_shared_f32(lse_s + c * 4));
        if (BIAS) arg = fmaf(bf16_bits_to_float(ld_shared_u16(bias_s + c * 256)), kLog2e, arg);
        float e = ex2_approx(arg);
        if (need_mask && c < first_vis) e = 0.f;
        pv[c] = e;
      }
      {
        // P~^T (bf16) into this step's S^T columns [0, 32) of TMEM
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 2 * c;
          float a = pv[e], bb = pv[e + 1];
          if (DROPOUT) {
            a = ((kb[e >> 5] >> (e & 31)) & 1u) ? a * p.drop_rescale : 0.f;
            bb = ((kb[(e + 1) >> 5] >> ((e + 1) & 31)) & 1u) ? bb * p.drop_rescale : 0.f;
          }
          pk[c] = pack_bf16x2(a, bb);
        }
        tmem_st32(tS, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&p_full[x]);

      mbar_wait_t<kInlineWaits>(&dp_full[x], k & 1, wc, kSiteBwdDpFull);
      tc_fence_after();
      if (k >= 1) mbar_wait_t<kInlineWaits>(&ds_empty[x], (k - 1) & 1, wc, kSiteBwdPdsEmpty);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
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
        if (BIAS && p.dbias.data != nullptr) {
          // dbias(i, kj) = dS(i, kj) replaces this thread's own bias column of
          // the stage tile (read above); the tile is stored by TMA below
#pragma unroll
          for (int i = 0; i < 32; ++i)
            st_shared_u16(bias_s + (cc * 32 + i) * 256, pack_bf16x2(ds[i], 0.f) & 0xffffu);
        }
        // dS^T (bf16 pairs along the query rows) to shared memory, the B
        // operand of dQ^T, and into S^T columns [32, 64) of TMEM (read
        // above), the A operand of dK: that product then reads no operand of
        // this step's from shared memory but Q
        uint32_t dsw[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c = cc * 4 + q4;  // 16-byte chunk along the 128-byte row
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dsw[4 * q4 + e] = pack_bf16x2(ds[8 * q4 + 2 * e], ds[8 * q4 + 2 * e + 1]);
          st_shared_v4(da + sw128_offset(r, c), dsw[4 * q4], dsw[4 * q4 + 1], dsw[4 * q4 + 2],
                       dsw[4 * q4 + 3]);
        }
        tmem_st16(tS + 32 + 16 * cc, dsw);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sp_empty[x]);
      fence_async_smem();
      mbar_arrive(&ds_full[x]);
      if (BIAS && p.dbias.data != nullptr) {
        // the warpgroup's dbias tile [MQ rows x 128 keys]; rows past Sq and
        // keys past Sk are clipped by the store
        named_barrier_sync(5 + x, 128);
        if (r == 0) {
          tma_store_4d(&tm_dbias, smem + L::kBiasT + st * L::kBiasBytes, k0, i0, h, b);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(&dbias_read[st]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ warpgroup (warps 8-11)
    const int lt = threadIdx.x - 256;  // TMEM lane = d
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t qa = sb + L::kDq;
    float* part = p.dq_part ? p.dq_part + static_cast<size_t>(kv_tile) * p.part_stride : nullptr;
    for (int t = 0; t < n_steps; ++t) {
      const int x = t & 1;
      const int i0 = (qt_first + t) * MQ;
      mbar_wait_t<kInlineWaits>(&dq_full[x], (t >> 1) & 1, wc, kSiteBwdDqFull);
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(tmem + L::tmem_dp(x) + lane_base, r0);
      tmem_ld32(tmem + L::tmem_dp(x) + lane_base + 32, r1);
      tmem_ld_wait(r0);
      touch32(r1);
      tc_fence_before();
      mbar_arrive(&dq_empty[x]);
      if (VARLEN && part == nullptr) {
        // Packed batches: each warp stages its own 32 columns (its TMEM
        // lanes) of the step's 64 rows, row-major [64][32] fp32 in its
        // quarter of the staging area, and reduce-adds them with one tiled
        // tensor reduce, so the four warps never wait for one another
        // (0.733 against 0.793 ms on the packed causal batch of mixed
        // lengths; 4 % slower than the bulk form on the long decoder).
        const int wq = lt >> 5;
        const uint32_t qw = qa + wq * (L::kDqBytes / 4);
        // (a 64-wide accumulator, head dims up to 64, has no columns for
        // warps 2 and 3: theirs are zeros)
        if (32 * wq < p.acc_w) {
          if (lane == 0) bulk_wait_read_all();  // this warp's previous reduce has read its quarter
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            st_shared_f32(qw + (c * 32 + lane) * 4, __uint_as_float(r0[c]));
            st_shared_f32(qw + ((32 + c) * 32 + lane) * 4, __uint_as_float(r1[c]));
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_2d(&tm_dq, smem + L::kDq + wq * (L::kDqBytes / 4), 32 * wq,
                              bh * p.Sq_pad + i0);
            bulk_commit();
          }
        }
      } else {
        // the whole tile, row-major [MQ][aw] fp32 with aw = 128, or 64 for
        // head dims up to 64, whose columns past 64 are zeros and are
        // neither staged nor reduced (aw a compile-time constant in each
        // branch: a runtime row width cost the 128-wide case 10 %); each
        // warp's first lane reduces (deterministic mode: stores into this
        // key tile's slice) a quarter of it, 16 rows, so four bulk
        // operations are in flight
        auto stage = [&](auto width) {
          constexpr int aw = decltype(width)::value;
          if ((lt & 31) == 0) bulk_wait_read_all();  // the previous copies have read the tile
          named_barrier_sync(2, 128);
          if (aw == 128 || lt < aw) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              st_shared_f32(qa + (c * aw + lt) * 4, __uint_as_float(r0[c]));
              st_shared_f32(qa + ((32 + c) * aw + lt) * 4, __uint_as_float(r1[c]));
            }
          }
          fence_async_smem();
          named_barrier_sync(2, 128);
          if ((lt & 31) == 0) {
            const int hh = lt >> 5;
            dq_out(p.dq_acc, part, (static_cast<size_t>(bh) * p.Sq_pad + i0 + 16 * hh) * aw,
                   smem + L::kDq + hh * 16 * aw * 4, 16 * aw * 4);
            bulk_commit();
          }
        };
        if (p.acc_w == 64)
          stage(std::integral_constant<int, 64>{});
        else
          stage(std::integral_constant<int, 128>{});
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
    // a packed sequence's last key tile is stored row by row, so that rows
    // of the next sequence are never written (uniform over the CTA)
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
        for (int s = 0; s < 2; ++s)  // column slabs the caller's head dim reaches
          if (s * 64 < p.D_io)
            tma_store_4d(is_dv ? &tm_dv : &tm_dk, smem + (is_dv ? L::kK : L::kV) + s * L::kKvSlab,
                         s * 64, ks + k0, h, tb);
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

template <bool C, bool DR, bool BI, bool VL>
cudaError_t launch_t(const CUtensorMap* m, const BwdParams& p, cudaStream_t stream) {
  auto kern = bwd_main_kernel_d128<C, DR, BI, VL>;
  const int smem = B128<BI>::kAlloc;
  cudaError_t e = ensure_smem_attr<bwd_main_kernel_d128<C, DR, BI, VL>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.n_kv_tiles) * static_cast<unsigned>(p.B * p.H);
  kern<<<grid, B128<BI>::kThreads, smem, stream>>>(m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7],
                                                   m[8], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_d128(bool causal, bool dropout, const CUtensorMap* maps,
                                 const BwdParams& p, cudaStream_t stream) {
  if (p.cu_q != nullptr) {  // packed batch (no bias)
    if (causal && dropout) return launch_t<true, true, false, true>(maps, p, stream);
    if (causal) return launch_t<true, false, false, true>(maps, p, stream);
    if (dropout) return launch_t<false, true, false, true>(maps, p, stream);
    return launch_t<false, false, false, true>(maps, p, stream);
  }
  if (p.bias.data != nullptr) {
    if (causal && dropout) return launch_t<true, true, true, false>(maps, p, stream);
    if (causal) return launch_t<true, false, true, false>(maps, p, stream);
    if (dropout) return launch_t<false, true, true, false>(maps, p, stream);
    return launch_t<false, false, true, false>(maps, p, stream);
  }
  if (causal && dropout) return launch_t<true, true, false, false>(maps, p, stream);
  if (causal) return launch_t<true, false, false, false>(maps, p, stream);
  if (dropout) return launch_t<false, true, false, false>(maps, p, stream);
  return launch_t<false, false, false, false>(maps, p, stream);
}

}  // namespace sdpa
