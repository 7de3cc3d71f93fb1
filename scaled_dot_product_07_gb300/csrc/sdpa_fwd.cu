// Forward kernel of fused scaled-dot-product attention for training
// (sdpfa_fwd of test_sdpa_loop_split, "DID loop split for SDPA", NVIDIA/Fuser
// PR 3711): out = dropout(softmax(scale * Q K^T + causal)) V and the
// natural-log log-sum-exp of each score row, stashed for the backward
// (NVIDIA/Fuser issue 2278, "SdpaOpFwd / SdpaOpBwd nodes").
//
// An item is two 128-row query tiles (Q0, Q1: 256 rows) of one (batch,
// head). Each CTA runs two items back to back (item c and item total-1-c:
// long causal tile pairs matched with short ones), 320 threads:
//   warp 9      TMA producer: per item Q0, Q1 (once the previous item's
//               last S product has read them), then K_j and V_j (separate
//               barriers) through a ring of 128-byte-swizzled stages that
//               runs on across items.
//   warp 8      TMEM allocator and MMA issuer (the warp runs converged, one
//               elected lane issues the tcgen05 instructions). TMEM holds
//               S0, S1 (128 fp32 columns each) and O0, O1 (D columns each).
//               Per key tile j it issues, in this order,
//                 O0 += P0_j V_j,  S0_{j+1} = Q0 K_{j+1}^T,
//                 O1 += P1_j V_j,  S1_{j+1} = Q1 K_{j+1}^T,
//               so that while the softmax works on one tile's scores the
//               tensor core runs the other tile's products (ping-pong).
//               P_i is bf16 written by the softmax into the first 64 columns
//               of S_i and is read straight from TMEM as the A operand.
//   warps 0-7   softmax, both warpgroups on the same tile (Q0's scores,
//               then Q1's): warps w and w+4 share TMEM lanes, so thread
//               (half, r) owns keys [64 half, 64 half + 64) of query row r.
//               Per key tile it loads its half row, masks the causal
//               diagonal / key tail, agrees on the row max with its partner
//               half (shared memory + 64-thread named barrier), rescales its
//               half of the O row in TMEM only when the max grew by more
//               than 2^8 (exact: the shift only changes the common
//               reference), and stores its half of P (bf16, dropout
//               applied) into TMEM. Halving the work per thread halves the
//               softmax latency each tile adds to the ping-pong. At the end
//               of an item the halves' row sums are combined and out = O / l
//               is stored straight from registers (the Q tiles are already
//               being refilled) and lse = m * scale + ln l written; the next
//               item's first products run meanwhile.
// The completion of S_i(j+1) implies that O_i += P_i(j) V_j has completed
// (tcgen05 operations of one issuing thread complete in order), so the
// softmax may touch O_i as soon as it sees its next scores.
// Key tiles entirely above the causal diagonal are never loaded or computed.
// Small grids (at most two items per SM) run one item per CTA.
//
// With an additive bias the forward is fwd_kernel_bias: the same roles and
// products, one item per CTA, plus a warp that loads each score tile's bias
// tile by TMA into a staging tile the softmax reads before its scores are
// ready; out staged in the dead Q tiles and stored by TMA.
//
// With dropout and a caller's keep-bit buffer (FwdParams::drop_bits), the
// STORE instantiation also writes each half row's 64 keep bits there for the
// backward; it draws them before exponentiating and applies them from the
// bits (its own instantiation, so that the plain dropout kernel's register
// allocation is untouched).
#include <type_traits>

#include "common.cuh"

namespace sdpa {
namespace {

template <int D>
struct FwdLayout {
  static constexpr int kSlabBytes = 128 * 128;            // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;          // 128 rows x D bf16
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr int kQ = 0;                            // Q0, Q1
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  // row-max / row-sum exchange between the two halves of a row:
  // [tile 2][parity 2][half 2][row 128] fp32
  static constexpr int kRed = kV + kStages * kTileBytes;
  static constexpr int kBar = kRed + 2 * 2 * 2 * 128 * 4;
  // q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], p_full[2], o_full[2]
  static constexpr int kNumBars = 1 + 4 * kStages + 6 + 1;  // + q_free
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;             // room to align to 1024
  // TMEM columns
  __host__ __device__ static constexpr uint32_t tmem_s(int i) { return 128u * i; }
  __host__ __device__ static constexpr uint32_t tmem_o(int i) { return 256u + D * i; }
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 320;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// The forward with a bias keeps the same Q, K and V tiles and adds a 32 KB
// staging tile for the bias of the next score tile: [half 2][row 128][128
// bytes], each half a 128-byte-swizzled TMA box of 64 keys, so that thread
// (half, row) finds its 64 values at row*128 + (chunk ^ (row & 7))*16 of its
// half and a warp's reads of one chunk hit distinct banks. To make room, the
// row-max exchange between the two halves of a row uses one slot per (half,
// row) instead of four.
template <int D>
struct FwdBiasLayout : FwdLayout<D> {
  using Base = FwdLayout<D>;
  static constexpr int kRed = Base::kRed;                 // [half 2][row 128] fp32
  static constexpr int kBar = kRed + 2 * 128 * 4;
  // the base set, then bias_full (the TMA has landed the staged tile) and
  // bias_empty (every softmax thread has read it)
  static constexpr int kNumBars = Base::kNumBars + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBiasStage = (kMisc + 16 + 1023) / 1024 * 1024;
  static constexpr int kBytes = kBiasStage + 256 * 128;
  static constexpr int kAlloc = kBytes + 1024;
  // softmax warps 0-7, MMA warp 8, TMA warp 9, bias TMA warp 10
  static constexpr int kThreads = 352;
  static_assert(kAlloc <= 232448, "shared memory budget");
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

// Number of key tiles that query rows [r0, r0+128) ∩ [0, Sq) can see.
__device__ __forceinline__ int kv_tiles_for(int r0, int Sq, int Sk, bool causal) {
  if (r0 >= Sq) return 0;
  const int n = (Sk + 127) / 128;
  if (!causal) return n;
  return min(n, min(r0 + 127, Sq - 1) / 128 + 1);
}

// One unit of work: a pair of 128-row query tiles of one (batch, head).
struct FwdItem {
  int b, h, bh, q0, Sq, Sk, qs, ks, tb;
  int n_t0, n_t1, n_kv;
  bool active;   // the tile pair holds query rows
  bool no_keys;  // a packed sequence with queries and no keys
};

// Head-major item order (a head's K/V stays in L2 while its items run); within
// a head the longest causal tile pairs come first.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int item) {
  FwdItem it;
  const int n_pairs = p.n_q_tiles;
  const int slot = item / n_pairs;
  int pair = item - slot * n_pairs;
  if (CAUSAL) pair = n_pairs - 1 - pair;
  // batch-major, or head-major when a bias shared by the batch makes the
  // batches of one head read the same bias tiles
  it.b = p.h_major ? slot % p.B : slot / p.H;
  it.h = p.h_major ? slot / p.B : slot - it.b * p.H;
  it.bh = it.b * p.H + it.h;
  it.q0 = pair * 256;
  // the sequence: the whole [Sq, Sk] problem, or sequence b of a packed batch
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
  it.tb = VARLEN ? 0 : it.b;  // batch coordinate in the tensor maps
  it.active = it.q0 < it.Sq;
  it.no_keys = it.active && it.Sk <= 0;
  const bool work = it.active && !it.no_keys;
  it.n_t0 = work ? kv_tiles_for(it.q0, it.Sq, it.Sk, CAUSAL) : 0;
  it.n_t1 = work ? kv_tiles_for(it.q0 + 128, it.Sq, it.Sk, CAUSAL) : 0;
  it.n_kv = max(it.n_t0, it.n_t1);
  return it;
}

// STORE (with DROPOUT, not VARLEN): the keep bits are also written to
// p.drop_bits for the backward. It is a separate instantiation so that the
// plain dropout kernel keeps its registers.
template <int D, bool CAUSAL, bool DROPOUT, bool VARLEN, bool STORE = false>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ FwdParams p) {
  using L = FwdLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + S;
  uint64_t* k_empty = v_full + S;
  uint64_t* v_empty = k_empty + S;
  uint64_t* s_full = v_empty + S;    // [2]
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* o_full = p_full + 2;     // [2]
  uint64_t* q_free = o_full + 2;     // every S product of an item has read Q0, Q1
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // CTA c runs item c and then item total-1-c: in the head-major order the
  // long causal tile pairs of one window are matched with the short ones of
  // the other, so every CTA gets about the same work, and the second item's
  // Q and first K/V tiles load while the first item finishes.
  const bool two = p.two_items != 0;
  const int total = p.n_q_tiles * p.B * p.H;
  const int first_item = blockIdx.x;
  const int second_item = two ? total - 1 - static_cast<int>(blockIdx.x) : 0;
  const int n_items = (two && second_item > first_item) ? 2 : 1;
  auto item_id = [&](int k) { return k == 0 ? first_item : second_item; };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 256);
      mbar_init(&o_full[i], 1);
    }
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

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      int qk = 0;  // Q loads issued (phases of q_full / q_free)
      int g = 0;   // K / V tiles issued over all items (ring position)
      for (int k = 0; k < n_items; ++k) {
        const FwdItem it = fwd_item<CAUSAL, VARLEN>(p, item_id(k));
        if (it.n_kv == 0) continue;
        // Q0, Q1 of the previous item are free once its last S product is done
        if (qk >= 1) mbar_wait(q_free, (qk - 1) & 1, wc, kSiteFwdQFull);
        const int nq = it.n_t1 > 0 ? 2 : 1;
        mbar_arrive_expect_tx(q_full, nq * L::kTileBytes);
        for (int i = 0; i < nq; ++i) {
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(smem + L::kQ + i * L::kTileBytes + s * L::kSlabBytes, &tm_q, q_full,
                        s * 64, it.qs + it.q0 + 128 * i, it.h, it.tb);
        }
        ++qk;
        for (int j = 0; j < it.n_kv; ++j, ++g) {
          const int st = g % S;
          // a K stage is free once the last S MMA reading it is done, a V stage
          // once the last P V MMA reading it is done
          if (g >= S) mbar_wait(&k_empty[st], ((g / S) - 1) & 1, wc, kSiteFwdKvEmpty);
          mbar_arrive_expect_tx(&k_full[st], L::kTileBytes);
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(smem + L::kK + st * L::kTileBytes + s * L::kSlabBytes, &tm_k, &k_full[st],
                        s * 64, it.ks + j * 128, it.h, it.tb);
          if (g >= S) mbar_wait(&v_empty[st], ((g / S) - 1) & 1, wc, kSiteFwdKvEmpty);
          mbar_arrive_expect_tx(&v_full[st], L::kTileBytes);
#pragma unroll
          for (int s = 0; s < D / 64; ++s)
            tma_load_4d(smem + L::kV + st * L::kTileBytes + s * L::kSlabBytes, &tm_v, &v_full[st],
                        s * 64, it.ks + j * 128, it.h, it.tb);
        }
      }
      if (*abort_word) {
        // give the loads still in flight time to land before the CTA exits
        for (int gg = max(0, g - S); gg < g; ++gg) {
          mbar_wait_drain(&k_full[gg % S], (gg / S) & 1, 2000000ull);
          mbar_wait_drain(&v_full[gg % S], (gg / S) & 1, 2000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and descriptor arithmetic are
    // warp-uniform); one elected lane issues the tcgen05 instructions.
    // Per key tile j it issues O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j,
    // S1 = Q1 K_{j+1}^T (ping-pong between the two query tiles).
    const uint32_t leader = elect_one();
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdO = idesc_bf16_f32(128, D, false, true);
    auto issue_s = [&](int i, int st) {
      const uint64_t qd = sdesc_sw128(sb + L::kQ + i * L::kTileBytes, 16, 1024);
      const uint64_t kd = sdesc_sw128(sb + L::kK + st * L::kTileBytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = (kk >> 2) * L::kSlabBytes + (kk & 3) * 32;
        mma_bf16_ss_if(leader, tmem + L::tmem_s(i), sdesc_add(qd, koff), sdesc_add(kd, koff), kIdS,
                       kk > 0 ? 1u : 0u);
      }
      mma_commit_if(leader, &s_full[i]);
    };
    auto issue_pv = [&](int i, int st, bool first) {
      const uint64_t vd = sdesc_sw128(sb + L::kV + st * L::kTileBytes, L::kSlabBytes, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16_ts_if(leader, tmem + L::tmem_o(i), tmem + L::tmem_s(i) + kk * 8,
                       sdesc_add(vd, kk * 2048), kIdO, (!first || kk > 0) ? 1u : 0u);
    };
    int qk = 0, g = 0;
    int pc[2] = {0, 0};  // P tiles consumed per query tile (phases of p_full)
    for (int k = 0; k < n_items; ++k) {
      const FwdItem it = fwd_item<CAUSAL, VARLEN>(p, item_id(k));
      if (it.n_kv == 0) continue;
      const int n_t[2] = {it.n_t0, it.n_t1};
      mbar_wait(q_full, qk & 1, wc, kSiteFwdQFull);
      ++qk;
      const int g0 = g;
      mbar_wait(&k_full[g0 % S], (g0 / S) & 1, wc, kSiteFwdKvFull);
      tc_fence_after();
      for (int i = 0; i < 2; ++i)
        if (n_t[i] > 0) issue_s(i, g0 % S);
      mma_commit_if(leader, &k_empty[g0 % S]);  // K_0 has no other reader
      if (it.n_kv == 1) mma_commit_if(leader, q_free);
      for (int j = 0; j < it.n_kv; ++j) {
        const int gj = g0 + j;
        const int st = gj % S;
        mbar_wait(&v_full[st], (gj / S) & 1, wc, kSiteFwdKvFull);
        for (int i = 0; i < 2; ++i) {
          if (j >= n_t[i]) continue;
          // P_i of this tile; it also orders the previous item's epilogue
          // reads of O_i before the first P V product overwrites O_i
          mbar_wait(&p_full[i], pc[i] & 1, wc, kSiteFwdPFull);
          ++pc[i];
          tc_fence_after();
          issue_pv(i, st, j == 0);
          if (j + 1 < n_t[i]) {
            const int g1 = gj + 1;
            mbar_wait(&k_full[g1 % S], (g1 / S) & 1, wc, kSiteFwdKvFull);
            tc_fence_after();
            issue_s(i, g1 % S);
          } else {
            mma_commit_if(leader, &o_full[i]);
          }
        }
        mma_commit_if(leader, &v_empty[st]);                                 // V_j read by both P V
        if (j + 1 < it.n_kv) mma_commit_if(leader, &k_empty[(gj + 1) % S]);  // K_{j+1} by both S
        if (j + 2 == it.n_kv) mma_commit_if(leader, q_free);  // the item's last S is issued
      }
      g += it.n_kv;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    // Both warpgroups work on the same tile: warp w and warp w+4 share TMEM
    // lanes, so thread (half, r) handles key columns [64h, 64h+64) of query row
    // r. The two halves of a row agree on its max through shared memory and
    // a 64-thread named barrier per warp pair; their partial row sums are
    // combined only at the end.
    const int half = warp >> 2;         // half of the key columns
    const int row = threadIdx.x & 127;  // row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t pair_bar = 1 + (warp & 3);  // + 4 * tile
    float* red = reinterpret_cast<float*>(smem + L::kRed);
    const float sl2 = p.scale_log2;
    const PhiloxKey pk = DROPOUT ? launch_key(p.pk, p.rng_dev) : p.pk;
    int sc[2] = {0, 0};  // S tiles consumed per query tile (phases of s_full)
    int oc[2] = {0, 0};  // items finished per query tile (phases of o_full)
    int xc[2] = {0, 0};  // exchanges per query tile; consecutive ones use alternate slots
    // this half's value v, shared with the partner half through the tile's
    // next exchange slot; returns the partner's value
    auto exchange = [&](int i, float v) {
      float* slot = red + ((i * 2 + (xc[i] & 1)) * 2) * 128;
      ++xc[i];
      slot[half * 128 + row] = v;
      // also orders the partner's TMEM score reads before this warp's P
      // stores into the same columns
      tc_fence_before();
      named_barrier_sync(pair_bar + 4 * i, 64);
      tc_fence_after();
      return slot[(1 - half) * 128 + row];
    };

    for (int k = 0; k < n_items; ++k) {
      const FwdItem it = fwd_item<CAUSAL, VARLEN>(p, item_id(k));
      if (!it.active) continue;
      const int b = it.b, h = it.h, bh = it.bh, q0 = it.q0, Sq = it.Sq, Sk = it.Sk, qs = it.qs;
      if (it.no_keys) {
        // no keys: the rows' outputs are 0 and their log-sum-exp is -inf
        for (int r = threadIdx.x; r < 256 && q0 + r < Sq; r += 256) {
          uint16_t* o = static_cast<uint16_t*>(p.out_io.data) + h * p.out_io.sH +
                        static_cast<int64_t>(qs + q0 + r) * p.out_io.sS;
          for (int c = 0; c < p.D_io; c += 8)
            *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
          p.lse[static_cast<size_t>(h) * p.total_q + qs + q0 + r] = -INFINITY;
        }
        continue;
      }
      const int n_t[2] = {it.n_t0, it.n_t1};
      float m[2] = {-INFINITY, -INFINITY};  // running max of the raw scores of the row, per tile
      float l[2] = {0.f, 0.f};              // this half's running sum, per tile
      for (int j = 0; j < it.n_kv; ++j) {
        for (int i = 0; i < 2; ++i) {
          if (j >= n_t[i]) continue;
          const int qi = q0 + 128 * i + row;
          const uint32_t tS = tmem + L::tmem_s(i) + lane_base;
          const uint32_t tO = tmem + L::tmem_o(i) + lane_base;
          // the non-causal dropout variants wait inline (2 % faster on the
          // encoder and cross-attention shapes); the causal ones out of
          // line (2 % slower inline on the long decoder)
          mbar_wait_t<!CAUSAL && DROPOUT>(&s_full[i], sc[i] & 1, wc, kSiteFwdSFull);
          ++sc[i];
          tc_fence_after();
          uint32_t r0[32], r1[32];
          tmem_ld32(tS + 64 * half, r0);
          tmem_ld32(tS + 64 * half + 32, r1);
          tmem_ld_wait(r0);
          reg_touch(r1);
          float x[64];
  #pragma unroll
          for (int c = 0; c < 32; ++c) {
            x[c] = __uint_as_float(r0[c]);
            x[32 + c] = __uint_as_float(r1[c]);
          }
          const int k0 = j * 128 + 64 * half;  // first key of this half
          if ((k0 + 64 > Sk) || (CAUSAL && k0 + 63 > q0 + 128 * i)) {
            const int lim = CAUSAL ? min(Sk - k0, qi - k0 + 1) : (Sk - k0);
  #pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c >= lim) x[c] = -INFINITY;
          }
          // half-row max as 8 independent chains, then combined
          float mp[8];
  #pragma unroll
          for (int u = 0; u < 8; ++u) mp[u] = fmaxf(x[2 * u], x[2 * u + 1]);
  #pragma unroll
          for (int c = 16; c < 64; c += 16)
  #pragma unroll
            for (int u = 0; u < 8; ++u) mp[u] = fmax3(mp[u], x[c + 2 * u], x[c + 2 * u + 1]);
          const float mh =
              fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], fmax3(mp[5], mp[6], mp[7])));
          const float m_new = fmaxf(m[i], fmaxf(mh, exchange(i, mh)));
          if (j == 0) {
            m[i] = m_new;
          } else if (__any_sync(0xffffffffu, (m_new - m[i]) * sl2 > 8.0f)) {
            // both halves of these rows take this branch (same rows, same maxima);
            // O_i += P_i(j-1) V has completed (S_i(j) completed after it)
            const float alpha = ex2_approx((m[i] - m_new) * sl2);
            l[i] *= alpha;
            m[i] = m_new;
            auto rescale = [&](int c) {  // 32 of this half's D/2 columns of O
              uint32_t o[32];
              tmem_ld32(tO + (D / 2) * half + c * 32, o);
              tmem_ld_wait(o);
  #pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(tO + (D / 2) * half + c * 32, o);
            };
            if constexpr (DROPOUT) {
              // not unrolled beside the Philox chains' registers (measured
              // faster there; unrolled is faster without dropout)
  #pragma unroll 1
              for (int c = 0; c < D / 64; ++c) rescale(c);
            } else {
  #pragma unroll
              for (int c = 0; c < D / 64; ++c) rescale(c);
            }
          }
          const float neg = -m[i] * sl2;

          // P = exp2(x*scale*log2e - m); with dropout P~ = keep ? P : 0, and the
          // 1/(1-p) is applied to O in the epilogue. The row sum takes P.
          float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 8 independent partial sums
          uint32_t pk2[32];
          // mode 0: no dropout; 1, 3: the half row starts on a group boundary
          // (Sk a multiple of 4), so group g_row + t holds keys 4t .. 4t+3 and
          // is drawn where those keys are exponentiated; 2: keep bits first
          auto exp_pack = [&](auto mode_c, uint64_t g_row, const uint32_t(&keep)[2]) {
            constexpr int kMode = decltype(mode_c)::value;
  #pragma unroll
            for (int c = 0; c < 64; c += 4) {
              float e[4];
  #pragma unroll
              for (int w = 0; w < 4; ++w) e[w] = ex2_approx(fmaf(x[c + w], sl2, neg));
              rs[(c >> 2) & 7] += (e[0] + e[1]) + (e[2] + e[3]);
              if constexpr (kMode == 1 || kMode == 3) {
                // 1: round keys from the kernel parameters; 3: from the key
                // read out of device memory
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
                for (int w = 0; w < 4; ++w)
                  e[w] = ((keep[(c + w) >> 5] >> ((c + w) & 31)) & 1u) ? e[w] : 0.f;
              }
              pk2[c >> 1] = pack_bf16x2(e[0], e[1]);
              pk2[(c >> 1) + 1] = pack_bf16x2(e[2], e[3]);
            }
          };
          const uint32_t no_bits[2] = {0xffffffffu, 0xffffffffu};
          if (!DROPOUT) {
            exp_pack(std::integral_constant<int, 0>{}, 0, no_bits);
          } else {
            const uint64_t n0 = (counter_bh(b, h, p.b0, p.h0, p.H_total) * p.Sq_ctr + qi) *
                                    static_cast<uint64_t>(p.Sk_ctr) +
                                k0;
            // STORE: kept for the backward, words k0/32 and k0/32 + 1 of row qi
            uint32_t* wp = STORE ? p.drop_bits +
                                       (static_cast<size_t>(bh) * p.bits_kw + (k0 >> 5)) * p.bits_rows +
                                       qi
                                 : nullptr;
            if ((p.Sk_ctr & 3) == 0) {
              if constexpr (STORE) {
                // the half row's 16 groups first (group t: keys 4t .. 4t+3),
                // stored, then applied from the bits
                uint32_t keep[2];
                if (p.rng_dev == nullptr)
                  keep_words_aligned<true>(n0 >> 2, p.drop_threshold, p.pk, p.rk, keep);
                else
                  keep_words_aligned<false>(n0 >> 2, p.drop_threshold, pk, p.rk, keep);
                wp[0] = keep[0];
                wp[p.bits_rows] = keep[1];
                exp_pack(std::integral_constant<int, 2>{}, 0, keep);
              } else {
                if (p.rng_dev == nullptr)
                  exp_pack(std::integral_constant<int, 1>{}, n0 >> 2, no_bits);
                else
                  exp_pack(std::integral_constant<int, 3>{}, n0 >> 2, no_bits);
              }
            } else {
              uint32_t keep[2];
              keep_bits<2>(n0, p.drop_threshold, pk, keep);
              if (STORE) {
                wp[0] = keep[0];
                wp[p.bits_rows] = keep[1];
              }
              exp_pack(std::integral_constant<int, 2>{}, 0, keep);
            }
          }
          // P (bf16 pairs) of keys [64h, 64h+64) -> S columns [32h, 32h+32); they
          // overwrite scores this warp pair has already read
          tmem_st32(tS + 32 * half, pk2);
          l[i] += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_full[i]);
        }
      }
      // ---------------------------------------------------------- epilogue
      for (int i = 0; i < 2; ++i) {
        if (n_t[i] == 0) continue;
        const int qi = q0 + 128 * i + row;
        const uint32_t tO = tmem + L::tmem_o(i) + lane_base;
        // the row sum is the sum of both halves
        const float l_row = l[i] + exchange(i, l[i]);
        mbar_wait(&o_full[i], oc[i] & 1, wc, kSiteFwdODone);
        ++oc[i];
        tc_fence_after();
        // 1/l, and the dropout rescale 1/(1-p) of the kept weights
        const float inv_l = (DROPOUT ? p.drop_rescale : 1.f) / l_row;
        // rows are stored straight from registers (the Q tiles are being
        // refilled for the next item); columns past D_io are padding
        uint16_t* orow = static_cast<uint16_t*>(p.out_io.data) + it.tb * p.out_io.sB +
                         h * p.out_io.sH + static_cast<int64_t>(qs + qi) * p.out_io.sS;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {  // this half's D/2 columns
          uint32_t o[32];
          tmem_ld32(tO + (D / 2) * half + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int col0 = (D / 2) * half + c * 32 + q4 * 8;
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
                qi] = m[i] * (sl2 * kLn2) + __logf(l_row);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// The forward with an additive bias: one item (query-tile pair) per CTA, O
// staged in the dead Q tiles and stored by TMA. The same algorithm as
// fwd_kernel; kept as its own kernel because with a bias it ran 1.19 ms
// against fwd_kernel's 1.38 (B8 H16 S4096 D128 causal, relative-position
// bias [1,H,S,S]). A warp of its own (warp 10) loads each score tile's bias
// by TMA into one staging tile, which the softmax reads and releases before
// its scores are ready: 0.61 ms, against 1.03 with each thread copying its
// own 128 bytes with cp.async. Packed batches take no bias, so it has no
// packed form.
template <int D, bool CAUSAL, bool DROPOUT>
__global__ void __launch_bounds__(352, 1)
    fwd_kernel_bias(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_bias, const FwdParams p) {
  constexpr bool BIAS = true;
  using L = FwdBiasLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + S;
  uint64_t* k_empty = v_full + S;
  uint64_t* v_empty = k_empty + S;
  uint64_t* s_full = v_empty + S;    // [2]
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* o_full = p_full + 2;     // [2]
  uint64_t* bias_full = bars + L::Base::kNumBars;
  uint64_t* bias_empty = bias_full + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* abort_word = reinterpret_cast<uint32_t*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // head-major order (a head's K/V stays in L2 while its tiles run);
  // within a head the longest causal tiles go first
  const int n_pairs = p.n_q_tiles;  // tile pairs per head
  const int slot = blockIdx.x / n_pairs;
  int pair = blockIdx.x - slot * n_pairs;
  if (CAUSAL) pair = n_pairs - 1 - pair;
  // (b, h) of this CTA: batch-major, or head-major when a bias shared by the
  // batch makes the batches of one head read the same bias tiles
  const int b = p.h_major ? slot % p.B : slot / p.H;
  const int h = p.h_major ? slot / p.B : slot - b * p.H;
  const int bh = b * p.H + h;
  const int q0 = pair * 256;
  const int Sq = p.Sq, Sk = p.Sk, qs = 0, ks = 0;
  const int tb = b;  // batch coordinate in the tensor maps
  const int n_t[2] = {kv_tiles_for(q0, Sq, Sk, CAUSAL), kv_tiles_for(q0 + 128, Sq, Sk, CAUSAL)};
  const int n_kv = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 256);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(bias_full, 1);
    mbar_init(bias_empty, 256);
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

  if (warp == 10) {
    // ------------------------------------------------------------ bias TMA
    // The bias tile of every score tile, in the order the softmax visits
    // them, into the one staging tile once the softmax has read the previous
    // one. Keys past Sk and rows past Sq read as zeros.
    if (lane == 0) {
      prefetch_tmap(&tm_bias);
      const int hb = p.bias.sH != 0 ? h : 0;
      const int bb = p.bias.sB != 0 ? b : 0;
      int t = 0;  // tiles loaded
      for (int j = 0; j < n_kv; ++j) {
        for (int i = 0; i < 2; ++i) {
          if (j >= n_t[i]) continue;
          if (t >= 1) mbar_wait(bias_empty, (t - 1) & 1, wc, kSiteFwdBiasEmpty);
          ++t;
          mbar_arrive_expect_tx(bias_full, 256 * 128);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_4d(smem + L::kBiasStage + hf * 128 * 128, &tm_bias, bias_full,
                        j * 128 + 64 * hf, q0 + 128 * i, hb, bb);
        }
      }
      if (*abort_word && t >= 1) mbar_wait_drain(bias_full, (t - 1) & 1, 2000000ull);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      const int nq = n_t[1] > 0 ? 2 : 1;
      mbar_arrive_expect_tx(q_full, nq * L::kTileBytes);
      for (int i = 0; i < nq; ++i) {
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(smem + L::kQ + i * L::kTileBytes + s * L::kSlabBytes, &tm_q, q_full, s * 64,
                      qs + q0 + 128 * i, h, tb);
      }
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        // a K stage is free once the last S MMA reading it is done, a V stage
        // once the last P V MMA reading it is done
        if (j >= S) mbar_wait(&k_empty[st], ((j / S) - 1) & 1, wc, kSiteFwdKvEmpty);
        mbar_arrive_expect_tx(&k_full[st], L::kTileBytes);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(smem + L::kK + st * L::kTileBytes + s * L::kSlabBytes, &tm_k, &k_full[st],
                      s * 64, ks + j * 128, h, tb);
        if (j >= S) mbar_wait(&v_empty[st], ((j / S) - 1) & 1, wc, kSiteFwdKvEmpty);
        mbar_arrive_expect_tx(&v_full[st], L::kTileBytes);
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_4d(smem + L::kV + st * L::kTileBytes + s * L::kSlabBytes, &tm_v, &v_full[st],
                      s * 64, ks + j * 128, h, tb);
      }
      if (*abort_word) {
        // give the loads still in flight time to land before the CTA exits
        for (int j = max(0, n_kv - S); j < n_kv; ++j) {
          mbar_wait_drain(&k_full[j % S], (j / S) & 1, 2000000ull);
          mbar_wait_drain(&v_full[j % S], (j / S) & 1, 2000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and descriptor arithmetic are
    // warp-uniform); one elected lane issues the tcgen05 instructions.
    const uint32_t leader = elect_one();
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdO = idesc_bf16_f32(128, D, false, true);
    auto issue_s = [&](int i, int j) {
      const int st = j % S;
      const uint64_t qd = sdesc_sw128(sb + L::kQ + i * L::kTileBytes, 16, 1024);
      const uint64_t kd = sdesc_sw128(sb + L::kK + st * L::kTileBytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = (kk >> 2) * L::kSlabBytes + (kk & 3) * 32;
        mma_bf16_ss_if(leader, tmem + L::tmem_s(i), sdesc_add(qd, koff), sdesc_add(kd, koff), kIdS,
                       kk > 0 ? 1u : 0u);
      }
      mma_commit_if(leader, &s_full[i]);
    };
    auto issue_pv = [&](int i, int j) {
      const int st = j % S;
      const uint64_t vd = sdesc_sw128(sb + L::kV + st * L::kTileBytes, L::kSlabBytes, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16_ts_if(leader, tmem + L::tmem_o(i), tmem + L::tmem_s(i) + kk * 8,
                       sdesc_add(vd, kk * 2048), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
    };
    mbar_wait(q_full, 0, wc, kSiteFwdQFull);
    if (n_kv > 0) {
      mbar_wait(&k_full[0], 0, wc, kSiteFwdKvFull);
      tc_fence_after();
      for (int i = 0; i < 2; ++i)
        if (n_t[i] > 0) issue_s(i, 0);
      mma_commit_if(leader, &k_empty[0]);  // K_0 has no other reader
    }
    for (int j = 0; j < n_kv; ++j) {
      const int st = j % S;
      mbar_wait(&v_full[st], (j / S) & 1, wc, kSiteFwdKvFull);
      for (int i = 0; i < 2; ++i) {
        if (j >= n_t[i]) continue;
        mbar_wait(&p_full[i], j & 1, wc, kSiteFwdPFull);
        tc_fence_after();
        issue_pv(i, j);
        if (j + 1 < n_t[i]) {
          const int st1 = (j + 1) % S;
          mbar_wait(&k_full[st1], ((j + 1) / S) & 1, wc, kSiteFwdKvFull);
          tc_fence_after();
          issue_s(i, j + 1);
        } else {
          mma_commit_if(leader, &o_full[i]);
        }
      }
      mma_commit_if(leader, &v_empty[st]);                             // V_j read by both P V
      if (j + 1 < n_kv) mma_commit_if(leader, &k_empty[(j + 1) % S]);  // K_{j+1} by both S
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    // Both warpgroups work on the same tile: warp w and warp w+4 share TMEM
    // lanes, so thread (half, r) handles key columns [64h, 64h+64) of query row
    // r. The two halves of a row agree on its max through shared memory and
    // a 64-thread named barrier per warp pair; their partial row sums are
    // combined only at the end.
    const int half = warp >> 2;         // half of the key columns
    const int row = threadIdx.x & 127;  // row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t pair_bar = 1 + (warp & 3);  // + 4 * tile
    float* red = reinterpret_cast<float*>(smem + L::kRed);
    const float sl2 = p.scale_log2;
    const PhiloxKey pk = DROPOUT ? launch_key(p.pk, p.rng_dev) : p.pk;
    float m[2] = {-INFINITY, -INFINITY};  // running max of the raw scores of the row, per tile
    float l[2] = {0.f, 0.f};              // this half's running sum, per tile
    // the half's value v, shared with the partner half through the pair's one
    // slot: the first barrier makes sure the partner has read the previous
    // value, the second that it has written this one
    auto exchange = [&](int i, float v) {
      named_barrier_sync(pair_bar + 4 * i, 64);
      red[half * 128 + row] = v;
      // also orders the partner's TMEM score reads before this warp's P
      // stores into the same columns
      tc_fence_before();
      named_barrier_sync(pair_bar + 4 * i, 64);
      tc_fence_after();
      return red[(1 - half) * 128 + row];
    };
    // the half's tile max, shared with the partner half; returns the row's tile max
    auto exchange_max = [&](int i, int j, float mh) {
      (void)j;
      return fmaxf(mh, exchange(i, mh));
    };
    // this thread's 64 bias values of the staged tile -- keys [j*128 + 64
    // half, +64) of row q0 + 128 i + row -- in its half's swizzled box
    const uint32_t bstage = sb + L::kBiasStage + (half * 128 + row) * 128;
    int bias_read = 0;  // bias tiles read

    for (int j = 0; j < n_kv; ++j) {
      for (int i = 0; i < 2; ++i) {
        if (j >= n_t[i]) continue;
        const int qi = q0 + 128 * i + row;
        const uint32_t tS = tmem + L::tmem_s(i) + lane_base;
        const uint32_t tO = tmem + L::tmem_o(i) + lane_base;
        // the staged bias tile, read and released before the scores are
        // ready, so that the next one loads while this tile is worked on
        uint4 bv[8];
        mbar_wait(bias_full, bias_read & 1, wc, kSiteFwdBiasFull);
        ++bias_read;
#pragma unroll
        for (int c = 0; c < 8; ++c) bv[c] = ld_shared_v4(bstage + ((c ^ (row & 7)) << 4));
        mbar_arrive(bias_empty);
        mbar_wait(&s_full[i], j & 1, wc, kSiteFwdSFull);
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(tS + 64 * half, r0);
        tmem_ld32(tS + 64 * half + 32, r1);
        tmem_ld_wait(r0);
        reg_touch(r1);
        float x[64];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0[c]);
          x[32 + c] = __uint_as_float(r1[c]);
        }
        if (BIAS) {
          // the bias in raw-score units (scores are scaled at the exponential)
          const float inv = p.bias_to_raw;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t w[4] = {bv[c].x, bv[c].y, bv[c].z, bv[c].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              x[8 * c + 2 * e] = fmaf(bf16_bits_to_float(w[e] & 0xffffu), inv, x[8 * c + 2 * e]);
              x[8 * c + 2 * e + 1] = fmaf(bf16_bits_to_float(w[e] >> 16), inv, x[8 * c + 2 * e + 1]);
            }
          }
        }
        const int k0 = j * 128 + 64 * half;  // first key of this half
        if ((k0 + 64 > Sk) || (CAUSAL && k0 + 63 > q0 + 128 * i)) {
          const int lim = CAUSAL ? min(Sk - k0, qi - k0 + 1) : (Sk - k0);
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c >= lim) x[c] = -INFINITY;
        }
        // half-row max as 8 independent chains, then combined
        float mp[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mp[u] = fmaxf(x[2 * u], x[2 * u + 1]);
#pragma unroll
        for (int c = 16; c < 64; c += 16)
#pragma unroll
          for (int u = 0; u < 8; ++u) mp[u] = fmax3(mp[u], x[c + 2 * u], x[c + 2 * u + 1]);
        const float mh =
            fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], fmax3(mp[5], mp[6], mp[7])));
        const float m_new = fmaxf(m[i], exchange_max(i, j, mh));
        if (j == 0) {
          m[i] = m_new;
        } else if (__any_sync(0xffffffffu, (m_new - m[i]) * sl2 > 8.0f)) {
          // both halves of these rows take this branch (same rows, same maxima);
          // O_i += P_i(j-1) V has completed (S_i(j) completed after it)
          const float alpha = ex2_approx((m[i] - m_new) * sl2);
          l[i] *= alpha;
          m[i] = m_new;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {  // this half's D/2 columns of O
            uint32_t o[32];
            tmem_ld32(tO + (D / 2) * half + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + (D / 2) * half + c * 32, o);
          }
        }
        const float neg = -m[i] * sl2;

        uint32_t keep[2] = {0xffffffffu, 0xffffffffu};
        if (DROPOUT) {
          const uint64_t n_row = (counter_bh(b, h, p.b0, p.h0, p.H_total) * p.Sq_ctr + qi) *
                                 static_cast<uint64_t>(p.Sk_ctr);
          keep_bits<2>(n_row + k0, p.drop_threshold, pk, keep);
        }
        // the same arithmetic as fwd_kernel: partial sums four keys at a time,
        // P~ = keep ? P : 0, and 1/(1-p) applied with 1/l in the epilogue
        float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 8 independent partial sums
        uint32_t pk2[32];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          float e[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) e[w] = ex2_approx(fmaf(x[c + w], sl2, neg));
          rs[(c >> 2) & 7] += (e[0] + e[1]) + (e[2] + e[3]);
          if (DROPOUT) {
#pragma unroll
            for (int w = 0; w < 4; ++w)
              e[w] = ((keep[(c + w) >> 5] >> ((c + w) & 31)) & 1u) ? e[w] : 0.f;
          }
          pk2[c >> 1] = pack_bf16x2(e[0], e[1]);
          pk2[(c >> 1) + 1] = pack_bf16x2(e[2], e[3]);
        }
        // P (bf16 pairs) of keys [64h, 64h+64) -> S columns [32h, 32h+32); they
        // overwrite scores this warp pair has already read
        tmem_st32(tS + 32 * half, pk2);
        l[i] += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[i]);
      }
    }

    // ------------------------------------------------------------ epilogue
    for (int i = 0; i < 2; ++i) {
      if (n_t[i] == 0) continue;
      const int qi = q0 + 128 * i + row;
      const uint32_t tO = tmem + L::tmem_o(i) + lane_base;
      // the row sum is the sum of both halves
      const float l_row = l[i] + exchange(i, l[i]);
      mbar_wait(&o_full[i], 0, wc, kSiteFwdODone);
      tc_fence_after();
      // 1/l, and the dropout rescale 1/(1-p) of the kept weights
      const float inv_l = (DROPOUT ? p.drop_rescale : 1.f) / l_row;
      const uint32_t oa = sb + L::kQ + i * L::kTileBytes;  // Q_i is dead after o_full[i]
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {  // this half's D/2 columns
        uint32_t o[32];
        tmem_ld32(tO + (D / 2) * half + c * 32, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int col0 = (D / 2) * half + c * 32 + q4 * 8;
          const uint32_t w0 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 0]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 1]) * inv_l);
          const uint32_t w1 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 3]) * inv_l);
          const uint32_t w2 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 4]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 5]) * inv_l);
          const uint32_t w3 = pack_bf16x2(__uint_as_float(o[q4 * 8 + 6]) * inv_l,
                                          __uint_as_float(o[q4 * 8 + 7]) * inv_l);
          st_shared_v4(oa + (col0 >> 6) * L::kSlabBytes + sw128_offset(row, (col0 & 63) >> 3),
                       w0, w1, w2, w3);
        }
      }
      if (half == 0 && qi < Sq)
        p.lse[static_cast<size_t>(bh) * Sq + qi] = m[i] * (sl2 * kLn2) + __logf(l_row);
      // rows past Sq and columns past D_io are clipped by the store
      fence_async_smem();
      named_barrier_sync(9 + i, 256);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_store_4d(&tm_o, smem + L::kQ + i * L::kTileBytes + s * L::kSlabBytes, s * 64,
                       qs + q0 + 128 * i, h, tb);
        bulk_commit();
        bulk_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}



// Two items per CTA once there are more than two items per SM, else one.
template <int D, bool C, bool DR, bool VL, bool ST = false>
cudaError_t launch_fwd_t(const CUtensorMap* maps, const FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_kernel<D, C, DR, VL, ST>;
  const int smem = FwdLayout<D>::kAlloc;
  cudaError_t e = ensure_smem_attr<fwd_kernel<D, C, DR, VL, ST>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned items = static_cast<unsigned>(p.n_q_tiles) * static_cast<unsigned>(p.B * p.H);
  FwdParams pl = p;
  pl.two_items = items > 2u * static_cast<unsigned>(device_sm_count());
  const unsigned grid = pl.two_items ? (items + 1) / 2 : items;
  kern<<<grid, FwdLayout<D>::kThreads, smem, stream>>>(maps[0], maps[1], maps[2], pl);
  return cudaGetLastError();
}

// One item per CTA.
template <int D, bool C, bool DR>
cudaError_t launch_fwd_bias_t(const CUtensorMap* maps, const FwdParams& p, cudaStream_t stream) {
  auto kern = fwd_kernel_bias<D, C, DR>;
  const int smem = FwdBiasLayout<D>::kAlloc;
  cudaError_t e = ensure_smem_attr<fwd_kernel_bias<D, C, DR>>(smem);
  if (e != cudaSuccess) return e;
  const unsigned items = static_cast<unsigned>(p.n_q_tiles) * static_cast<unsigned>(p.B * p.H);
  kern<<<items, FwdBiasLayout<D>::kThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                            maps[4], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, bool causal, bool dropout, const CUtensorMap* maps,
                       const FwdParams& p, cudaStream_t stream) {
  const bool bias = p.bias.data != nullptr;
  const bool varlen = p.cu_q != nullptr;  // packed batches take no bias
  // the keep bits are stored (dropout only; the host allows no bias, no
  // packed batch with them)
  const bool store = dropout && p.drop_bits != nullptr;
#define SDPA_FWD_CASE(DD, CC, RR)                                                    \
  if (D == DD && causal == CC && dropout == RR)                                      \
    return varlen ? launch_fwd_t<DD, CC, RR, true>(maps, p, stream)                  \
                  : (bias ? launch_fwd_bias_t<DD, CC, RR>(maps, p, stream)           \
                          : (store && RR ? launch_fwd_t<DD, CC, RR, false, RR>(maps, p, stream) \
                                         : launch_fwd_t<DD, CC, RR, false>(maps, p, stream)));
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
