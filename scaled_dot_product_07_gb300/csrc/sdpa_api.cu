// C-ABI entry points (include/sdpa.h): argument validation, TMA tensor maps
// for the caller's strided [B,H,S,D] tensors, and kernel launches on the
// caller's stream. The library allocates no device memory.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/sdpa.h"
#include "common.cuh"

namespace sdpa {
namespace {

// Device error word: the first bounded wait that gives up records its site.
__device__ uint32_t g_wait_error;

// ------------------------------------------------------------ small kernels

// Keep mask of a [B, H, Sq, Sk] block whose batches and heads start at
// (b0, h0) of a problem with H_total heads per batch.
__global__ void __launch_bounds__(256) dropout_mask_kernel(int64_t total, int64_t per_head, int H,
                                                           int b0, int h0, int H_total,
                                                           uint32_t threshold, PhiloxKey pk_arg,
                                                           const uint64_t* rng_dev, uint8_t* mask) {
  const PhiloxKey pk = launch_key(pk_arg, rng_dev);
  for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < total;
       n += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t bh = n / per_head;
    const int b = static_cast<int>(bh / H);
    const int h = static_cast<int>(bh - static_cast<int64_t>(b) * H);
    const uint64_t g = counter_bh(b, h, b0, h0, H_total) * static_cast<uint64_t>(per_head) +
                       static_cast<uint64_t>(n - bh * per_head);
    mask[n] = keep_one(g, threshold, pk) ? 1 : 0;
  }
}

__global__ void selftest_wait_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_word = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{&abort_word, err, limit_ns};
    mbar_wait(&bar, 0, wc, kSiteSelftest);  // nothing arrives: gives up after limit_ns
  }
  __syncthreads();
}

// ------------------------------------------------------------ host helpers

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Device address of g_wait_error on the current device (looked up once per
// device under a lock, with that device current). nullptr on failure.
uint32_t* error_word() {
  static uint32_t* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wait_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* e = std::getenv("SDPA_WAIT_LIMIT_MS");
    double ms = e ? std::atof(e) : 2000.0;
    if (!(ms > 0.0)) ms = 2000.0;
    return static_cast<uint64_t>(ms * 1e6);
  }();
  return v;
}

bool debug_sync() {
  static bool v = [] {
    const char* e = std::getenv("SDPA_DEBUG_SYNC");
    return e && e[0] == '1';
  }();
  return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape of one tensor argument, checked against expected [B,H,S,D].
sdpa_status check_tensor(const sdpa_tensor* t, int64_t B, int64_t H, int64_t S, int64_t D) {
  if (!t) return SDPA_ERR_INVALID_ARG;
  if (t->size[0] != B || t->size[1] != H || t->size[2] != S || t->size[3] != D)
    return SDPA_ERR_INVALID_ARG;
  const int64_t numel = B * H * S * D;
  if (numel == 0) return SDPA_OK;
  if (!t->data) return SDPA_ERR_INVALID_ARG;
  if (t->stride[3] != 1 && D > 1) return SDPA_ERR_UNSUPPORTED;
  for (int d = 0; d < 3; ++d) {
    if (t->size[d] > 1) {
      if (t->stride[d] <= 0) return SDPA_ERR_INVALID_ARG;
      if ((t->stride[d] * 2) % 16 != 0) return SDPA_ERR_ALIGNMENT;
    }
  }
  if (!aligned16(t->data)) return SDPA_ERR_ALIGNMENT;
  return SDPA_OK;
}

sdpa_status check_dims(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v) {
  if (!q || !k || !v) return SDPA_ERR_INVALID_ARG;
  for (int d = 0; d < 4; ++d)
    if (q->size[d] < 0 || k->size[d] < 0 || v->size[d] < 0) return SDPA_ERR_INVALID_ARG;
  const int64_t B = q->size[0], H = q->size[1], Sk = k->size[2];
  if (k->size[0] != B || k->size[1] != H || v->size[0] != B || v->size[1] != H ||
      v->size[2] != Sk)
    return SDPA_ERR_INVALID_ARG;
  // E = Ev: q, k and v share the head dim
  if (k->size[3] != q->size[3] || v->size[3] != q->size[3]) return SDPA_ERR_INVALID_ARG;
  const int64_t lim = int64_t(1) << 30;
  if (B > lim || H > lim || q->size[2] > lim || Sk > lim || B * H > lim)
    return SDPA_ERR_UNSUPPORTED;
  return SDPA_OK;
}

sdpa_status check_common(double p, float scale) {
  if (!(p >= 0.0 && p < 1.0)) return SDPA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return SDPA_ERR_INVALID_ARG;
  return SDPA_OK;
}

// 4-D tensor map over the logical dims (D, S, H, B), 128-byte swizzle,
// box = 64 elements (128 bytes) x box_rows rows.
bool make_map(CUtensorMap* m, const sdpa_tensor* t, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(t->size[3]), static_cast<cuuint64_t>(t->size[2]),
                        static_cast<cuuint64_t>(t->size[1]), static_cast<cuuint64_t>(t->size[0])};
  cuuint64_t strides[3];
  const int logical[3] = {2, 1, 0};  // S, H, B
  for (int k = 0; k < 3; ++k) {
    const int d = logical[k];
    int64_t sbytes = t->stride[d] * 2;
    if (t->size[d] <= 1) sbytes = 16;  // unused extent: any valid stride
    strides[k] = static_cast<cuuint64_t>(sbytes);
  }
  cuuint32_t box[4] = {64, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t->data, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map of the fp32 dQ accumulator as a [rows, 128] matrix (rows =
// B*H*Sq_pad): box [64 rows x 32 columns], the columns one dQ warp of the
// backward holds for a 64-row query step; no swizzle.
bool make_dq_map(CUtensorMap* m, float* acc, int64_t rows, int64_t width) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(width * 4)};
  cuuint32_t box[2] = {32, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, acc, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map of an attention bias (or its gradient) [Bb, Hb, Sq, Sk] (keys
// contiguous), zeros past the edges: the backward's box is [64 query rows x
// 128 keys] unswizzled (fwd = false), the forward's [128 query rows x 64
// keys] with the 128-byte swizzle (fwd = true). A shared dim (size 1 or
// stride 0) is always read at coordinate 0, so it gets a packed stride.
bool make_bias_map(CUtensorMap* m, const AttnBias& bias, int64_t Bb, int64_t Hb, int64_t Sq,
                   int64_t Sk, bool fwd = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  // a shared dim (size 1 or stride 0) is one slice, read at coordinate 0
  if (bias.sB == 0) Bb = 1;
  if (bias.sH == 0) Hb = 1;
  const int64_t rowS = Sq == 1 ? (Sk + 7) / 8 * 8 : bias.sS;
  const int64_t headS = Hb == 1 ? rowS * Sq : bias.sH;
  const int64_t batchS = Bb == 1 ? headS * Hb : bias.sB;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(Sk), static_cast<cuuint64_t>(Sq),
                        static_cast<cuuint64_t>(Hb), static_cast<cuuint64_t>(Bb)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(rowS * 2), static_cast<cuuint64_t>(headS * 2),
                           static_cast<cuuint64_t>(batchS * 2)};
  cuuint32_t box[4] = {fwd ? 64u : 128u, fwd ? 128u : 64u, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(bias.data), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fwd ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

PhiloxKey philox_key(uint64_t seed, uint64_t offset) {
  PhiloxKey k;
  k.k0 = static_cast<uint32_t>(seed);
  k.k1 = static_cast<uint32_t>(seed >> 32);
  k.off_lo = static_cast<uint32_t>(offset);
  k.off_hi = static_cast<uint32_t>(offset >> 32);
  return k;
}

uint32_t drop_threshold(double p) {
  const double t = std::floor(p * 4294967296.0);
  return t >= 4294967295.0 ? 0xFFFFFFFFu : static_cast<uint32_t>(t);
}

StridedBf16 strided(const sdpa_tensor* t) {
  return StridedBf16{t->data, t->stride[0], t->stride[1], t->stride[2]};
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// a*b*c*d fp32 words in bytes (all factors positive), or SIZE_MAX when that
// does not fit in 62 bits: no workspace satisfies such a request
size_t checked_bytes(int64_t a, int64_t b, int64_t c, int64_t d) {
  if (static_cast<double>(a) * static_cast<double>(b) * static_cast<double>(c) *
          static_cast<double>(d) * 4.0 >= 4.6e18)
    return SIZE_MAX;
  return static_cast<size_t>(a * b * c * d * 4);
}

// Head dims served: multiples of 8 up to 256. The forward kernels are built
// for 64, 128 and 256; a smaller D runs the next larger one, with the missing
// columns of q, k, v, dout read as zeros by the TMA loads (out-of-bounds
// fill) and never written by the stores. Zero columns add nothing to Q K^T,
// dO V^T or any product, so the results are those of the unpadded problem.
bool head_dim_supported(int64_t D) { return D >= 8 && D <= 256 && D % 8 == 0; }
int64_t kernel_head_dim(int64_t D) { return D <= 64 ? 64 : (D <= 128 ? 128 : 256); }
// The backward runs every head dim up to 128 on the 128-wide kernel: at D=64
// it beat a 64-wide kernel of 128-row query steps (B8 H16 S4096 causal: 1.31
// against 1.41 ms; with dropout 0.1: 2.05 against 4.53 ms). Larger head dims
// run the 256-wide kernel. The fp32 dQ rows of the workspace are as wide as
// the kernel's head dim.
int64_t bwd_kernel_head_dim(int64_t D) { return D <= 128 ? 128 : 256; }

// Columns of the backward's fp32 dQ accumulator: the kernel's width, except
// that head dims up to 64 (run on the 128-wide kernel, whose dQ columns past
// 64 are zeros) keep only 64, which halves the bytes its zero-fill, its
// reduce-adds and its conversion move.
int64_t dq_acc_width(int64_t D) { return D <= 64 ? 64 : bwd_kernel_head_dim(D); }

// Resolved sdpa_options.
struct Opts {
  const uint64_t* rng = nullptr;
  int b0 = 0, h0 = 0, H_total = 0;
  bool det = false;
  AttnBias bias{nullptr, 0, 0, 0};
  int64_t bias_B = 0, bias_H = 0;  // the bias's own batch and head extents (1 when shared)
  DBias dbias{nullptr, 0, 0, 0};
  cudaEvent_t ev_begin = nullptr, ev_end = nullptr;  // around the main kernel
  uint32_t* bits = nullptr;  // dropout keep bits carried from forward to backward
};

// Records one of the caller's kernel events (none when it is null).
cudaError_t record_event(cudaEvent_t ev, cudaStream_t stream) {
  return ev ? cudaEventRecord(ev, stream) : cudaSuccess;
}

sdpa_status check_bias(const sdpa_tensor* t, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                       AttnBias* out) {
  if (!t->data) return SDPA_ERR_INVALID_ARG;
  if ((t->size[0] != 1 && t->size[0] != B) || (t->size[1] != 1 && t->size[1] != H) ||
      t->size[2] != Sq || t->size[3] != Sk)
    return SDPA_ERR_INVALID_ARG;
  for (int d = 0; d < 4; ++d)
    if (t->stride[d] < 0) return SDPA_ERR_INVALID_ARG;
  if (Sk > 1 && t->stride[3] != 1) return SDPA_ERR_UNSUPPORTED;
  const int64_t sB = t->size[0] == 1 ? 0 : t->stride[0];
  const int64_t sH = t->size[1] == 1 ? 0 : t->stride[1];
  const int64_t sS = Sq == 1 ? 0 : t->stride[2];
  // 16-byte vector loads of 8 keys
  if ((reinterpret_cast<uintptr_t>(t->data) & 15u) || (sB % 8) || (sH % 8) || (sS % 8))
    return SDPA_ERR_ALIGNMENT;
  *out = AttnBias{static_cast<const uint16_t*>(t->data), sB, sH, sS};
  return SDPA_OK;
}

sdpa_status check_dbias(const sdpa_tensor* t, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                        DBias* out) {
  if (!t->data) return SDPA_ERR_INVALID_ARG;
  if (t->size[0] != B || t->size[1] != H || t->size[2] != Sq || t->size[3] != Sk)
    return SDPA_ERR_INVALID_ARG;
  for (int d = 0; d < 4; ++d)
    if (t->stride[d] < 0) return SDPA_ERR_INVALID_ARG;
  if (Sk > 1 && t->stride[3] != 1) return SDPA_ERR_UNSUPPORTED;
  // stored by TMA tiles: 16-byte aligned base and row, head, batch strides
  if ((reinterpret_cast<uintptr_t>(t->data) & 15u) || (t->stride[0] % 8) || (t->stride[1] % 8) ||
      (Sq > 1 && t->stride[2] % 8))
    return SDPA_ERR_ALIGNMENT;
  *out = DBias{static_cast<uint16_t*>(t->data), t->stride[0], t->stride[1], t->stride[2]};
  return SDPA_OK;
}

sdpa_status resolve_options(const sdpa_options* o, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                            Opts* r) {
  Opts x;
  x.H_total = static_cast<int>(H);
  // the launch grids number the 128-row query and key tiles of every (batch,
  // head) in int (sizes of real tensors stay far below this; views with
  // overlapping strides need not)
  const double tiles = static_cast<double>(B) * static_cast<double>(H) *
                       static_cast<double>((std::max(Sq, Sk) + 127) / 128);
  if (tiles > 2147483647.0) return SDPA_ERR_UNSUPPORTED;
  // the global counter ((b*H_total + h)*Sq + i)*Sk + j must fit in 64 bits
  auto counter_fits = [&](int64_t b_end, int64_t h_total) {
    return static_cast<double>(b_end) * static_cast<double>(h_total) * static_cast<double>(Sq) *
               static_cast<double>(Sk) < 1.8e19;
  };
  if (!counter_fits(B, H)) return SDPA_ERR_INVALID_ARG;
  if (o) {
    if (o->batch_offset < 0 || o->head_offset < 0 || o->total_heads < 0)
      return SDPA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(o->rng_state) & 7u) return SDPA_ERR_ALIGNMENT;
    const int64_t Ht = o->total_heads ? o->total_heads : H;
    if (o->head_offset + H > Ht) return SDPA_ERR_INVALID_ARG;
    const int64_t kMaxInt = 0x7fffffff;
    if (o->batch_offset + B > kMaxInt || Ht > kMaxInt) return SDPA_ERR_INVALID_ARG;
    if (!counter_fits(o->batch_offset + B, Ht)) return SDPA_ERR_INVALID_ARG;
    if (o->attn_bias) {
      const sdpa_status s = check_bias(o->attn_bias, B, H, Sq, Sk, &x.bias);
      if (s != SDPA_OK) return s;
      x.bias_B = o->attn_bias->size[0];
      x.bias_H = o->attn_bias->size[1];
    }
    if (o->dbias) {
      if (!o->attn_bias) return SDPA_ERR_INVALID_ARG;
      const sdpa_status s = check_dbias(o->dbias, B, H, Sq, Sk, &x.dbias);
      if (s != SDPA_OK) return s;
    }
    if (o->kernel_events) {
      x.ev_begin = static_cast<cudaEvent_t>(o->kernel_events[0]);
      x.ev_end = static_cast<cudaEvent_t>(o->kernel_events[1]);
      if (!x.ev_begin || !x.ev_end) return SDPA_ERR_INVALID_ARG;
    }
    if (o->dropout_bits) {
      if (reinterpret_cast<uintptr_t>(o->dropout_bits) & 3u) return SDPA_ERR_ALIGNMENT;
      if (o->dropout_bits_bytes < sdpa_dropout_bits_size(B, H, Sq, Sk)) return SDPA_ERR_INVALID_ARG;
      x.bits = o->dropout_bits;
    }
    x.rng = o->rng_state;
    x.b0 = static_cast<int>(o->batch_offset);
    x.h0 = static_cast<int>(o->head_offset);
    x.H_total = static_cast<int>(Ht);
    x.det = o->deterministic != 0;
  }
  *r = x;
  return SDPA_OK;
}

// Stored dropout bits serve the 128-wide kernels of one [Sq, Sk] problem per
// (batch, head): not the 256-wide ones, a bias or a packed batch.
sdpa_status check_bits(const Opts& opt, int64_t D, double dropout_p, bool packed) {
  if (opt.bits == nullptr || !(dropout_p > 0.0)) return SDPA_OK;
  if (D > 128 || opt.bias.data != nullptr || packed) return SDPA_ERR_UNSUPPORTED;
  return SDPA_OK;
}

sdpa_status finish(cudaError_t e, cudaStream_t stream) {
  if (e != cudaSuccess) return SDPA_ERR_CUDA;
  if (debug_sync()) return sdpa_check_device(reinterpret_cast<sdpa_stream_t>(stream));
  return SDPA_OK;
}

// A packed batch: B >= 1 sequences whose offsets are device arrays; the
// tensors are logical [1, H, total, D]. The offsets themselves are not read
// here (they live in device memory): they must start at 0, not decrease,
// end at the tensors' totals and give lengths of at most the maxima.
sdpa_status check_varlen(const sdpa_varlen* seqs, const sdpa_tensor* q, const sdpa_tensor* k) {
  if (!seqs || !seqs->cu_seqlens_q || !seqs->cu_seqlens_k) return SDPA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqs->cu_seqlens_q) & 3u) ||
      (reinterpret_cast<uintptr_t>(seqs->cu_seqlens_k) & 3u))
    return SDPA_ERR_ALIGNMENT;
  if (seqs->batch < 1 || seqs->max_seqlen_q < 1 || seqs->max_seqlen_k < 1) return SDPA_ERR_INVALID_ARG;
  if (seqs->batch > 0x7fffffff || seqs->max_seqlen_q > 0x7fffffff || seqs->max_seqlen_k > 0x7fffffff)
    return SDPA_ERR_INVALID_ARG;
  if (q->size[0] != 1 || k->size[0] != 1) return SDPA_ERR_INVALID_ARG;
  if (q->size[2] > 0x7fffffff || k->size[2] > 0x7fffffff) return SDPA_ERR_INVALID_ARG;
  return SDPA_OK;
}

// Shared tail of the forward entry points: tensor maps, parameters, launch.
// B, Sq, Sk are the problem's (or, packed, the batch count and the maximum
// lengths); cu_q / cu_k are null unless the batch is packed.
sdpa_status fwd_launch(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                       sdpa_tensor* out, float* lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                       int64_t D, double dropout_p, int is_causal, float scale, uint64_t seed,
                       uint64_t offset, const Opts& opt, const int32_t* cu_q, const int32_t* cu_k,
                       int64_t total_q, cudaStream_t stream) {
  const int64_t Dk = kernel_head_dim(D);
  // the 256-wide forward streams 64-key K / V tiles
  const uint32_t kv_rows = Dk == 256 ? 64 : 128;
  // q, k, v, out, bias (a copy of q's when there is none)
  CUtensorMap maps[5];
  if (!make_map(&maps[0], q, 128) || !make_map(&maps[1], k, kv_rows) ||
      !make_map(&maps[2], v, kv_rows) || !make_map(&maps[3], out, 128))
    return SDPA_ERR_CUDA;
  maps[4] = maps[0];
  if (opt.bias.data != nullptr &&
      !make_bias_map(&maps[4], opt.bias, opt.bias_B, opt.bias_H, Sq, Sk, true))
    return SDPA_ERR_CUDA;
  FwdParams p;
  p.B = static_cast<int>(B);
  p.H = static_cast<int>(H);
  p.Sq = static_cast<int>(Sq);
  p.Sk = static_cast<int>(Sk);
  // pairs of 128-row query tiles (one 128-row tile per CTA at D = 256)
  p.n_q_tiles = static_cast<int>(Dk == 256 ? (Sq + 127) / 128 : (Sq + 255) / 256);
  p.scale_log2 = scale * kLog2e;
  p.drop_threshold = drop_threshold(dropout_p);
  p.drop_rescale = static_cast<float>(1.0 / (1.0 - dropout_p));
  p.pk = philox_key(seed, offset);
  p.rk = philox_round_keys(p.pk);
  p.rng_dev = opt.rng;
  p.b0 = opt.b0;
  p.h0 = opt.h0;
  p.H_total = opt.H_total;
  p.bias = opt.bias;
  p.bias_to_raw = 1.0f / scale;
  p.h_major = (opt.bias.data != nullptr && opt.bias.sB == 0 && B > 1) ? 1 : 0;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.Sq_ctr = static_cast<int>(Sq);
  p.Sk_ctr = static_cast<int>(Sk);
  p.total_q = static_cast<int>(total_q);
  p.drop_bits = dropout_p > 0.0 ? opt.bits : nullptr;
  p.bits_kw = round_up(Sk, 128) / 32;
  p.bits_rows = round_up(Sq, 128);
  if (p.drop_bits != nullptr && (Dk == 256 || opt.bias.data != nullptr || cu_q != nullptr))
    return SDPA_ERR_UNSUPPORTED;
  p.D_io = static_cast<int>(D);
  p.out_io = strided(out);
  p.lse = lse;
  p.err = error_word();
  p.wait_limit_ns = wait_limit_ns();
  if (!p.err) return SDPA_ERR_CUDA;
  const bool dropout = dropout_p > 0.0;
  cudaError_t e = record_event(opt.ev_begin, stream);
  if (e == cudaSuccess)
    e = Dk == 256 ? launch_fwd_d256(is_causal != 0, dropout, maps, p, stream)
                  : launch_fwd(static_cast<int>(Dk), is_causal != 0, dropout, maps, p, stream);
  if (e == cudaSuccess) e = record_event(opt.ev_end, stream);
  return finish(e, stream);
}

// Shared tail of the backward entry points: workspace, tensor maps, the
// preprocess, main and dQ kernels. B, Sq, Sk are the problem's (or, packed,
// the batch count and the maximum lengths); cu_q / cu_k are null unless the
// batch is packed.
sdpa_status bwd_launch(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                       const sdpa_tensor* v, const sdpa_tensor* out, const float* lse, int64_t B,
                       int64_t H, int64_t Sq, int64_t Sk, int64_t D, double dropout_p,
                       int is_causal, uint64_t seed, uint64_t offset, float scale, sdpa_tensor* dq,
                       sdpa_tensor* dk, sdpa_tensor* dv, void* workspace, size_t workspace_bytes,
                       const sdpa_options* options, const Opts& opt, const int32_t* cu_q,
                       const int32_t* cu_k, int64_t total_q, cudaStream_t stream) {
  const int64_t Dk = bwd_kernel_head_dim(D);
  if (dropout_p > 0.0 && opt.bits != nullptr &&
      (Dk == 256 || opt.bias.data != nullptr || cu_q != nullptr))
    return SDPA_ERR_UNSUPPORTED;
  const size_t need = sdpa_bwd_workspace_size_ex(B, H, Sq, Sk, D, options);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SDPA_ERR_WORKSPACE;

  // workspace: [dQ accumulator | per-key-tile dQ partials (deterministic)], lse2, delta
  const int64_t Sq_pad = round_up(Sq, 128);
  const int64_t n_kv = (Sk + 127) / 128;
  const int64_t Da = dq_acc_width(D);
  const int64_t slice = B * H * Sq_pad * Da;
  float* dq_region = static_cast<float*>(workspace);
  float* lse2 = dq_region + slice * (opt.det ? n_kv : 1);
  float* delta = lse2 + B * H * Sq_pad;
  float* dq_acc = opt.det ? nullptr : dq_region;

  const uint32_t mq = static_cast<uint32_t>(8192 / Dk);
  // q, k, v, dout, dk, dv, bias, dbias, dq accumulator (copies of q's when absent)
  CUtensorMap maps[9];
  if (!make_map(&maps[0], q, mq) || !make_map(&maps[1], k, 128) || !make_map(&maps[2], v, 128) ||
      !make_map(&maps[3], dout, mq) || !make_map(&maps[4], dk, 128) || !make_map(&maps[5], dv, 128))
    return SDPA_ERR_CUDA;
  maps[6] = maps[0];
  maps[7] = maps[0];
  maps[8] = maps[0];
  // the packed-batch form of the 128-wide kernel reduces dQ through a 2-D map
  if (Dk == 128 && dq_acc != nullptr && !make_dq_map(&maps[8], dq_acc, B * H * Sq_pad, Da))
    return SDPA_ERR_CUDA;
  if (opt.bias.data != nullptr &&
      !make_bias_map(&maps[6], opt.bias, opt.bias_B, opt.bias_H, Sq, Sk))
    return SDPA_ERR_CUDA;
  if (opt.dbias.data != nullptr &&
      !make_bias_map(&maps[7], AttnBias{opt.dbias.data, opt.dbias.sB, opt.dbias.sH, opt.dbias.sS},
                     B, H, Sq, Sk))
    return SDPA_ERR_CUDA;

  uint32_t* err = error_word();
  if (!err) return SDPA_ERR_CUDA;

  PreParams pp;
  pp.B = static_cast<int>(B);
  pp.H = static_cast<int>(H);
  pp.Sq = static_cast<int>(Sq);
  pp.Sq_pad = static_cast<int>(Sq_pad);
  pp.D = static_cast<int>(Da);
  pp.D_io = static_cast<int>(D);
  pp.out = strided(out);
  pp.dout = strided(dout);
  pp.lse = lse;
  pp.lse2 = lse2;
  pp.delta = delta;
  pp.dq_acc = dq_acc;
  pp.cu_q = cu_q;
  pp.total_q = static_cast<int>(total_q);
  cudaError_t e = launch_bwd_preprocess(pp, stream);
  if (e != cudaSuccess) return SDPA_ERR_CUDA;

  BwdParams p;
  p.B = pp.B;
  p.H = pp.H;
  p.Sq = pp.Sq;
  p.Sk = static_cast<int>(Sk);
  p.Sq_pad = pp.Sq_pad;
  p.n_kv_tiles = static_cast<int>((Sk + 127) / 128);
  p.scale_log2 = scale * kLog2e;
  p.scale = scale;
  p.drop_threshold = drop_threshold(dropout_p);
  p.drop_rescale = static_cast<float>(1.0 / (1.0 - dropout_p));
  p.pk = philox_key(seed, offset);
  p.rng_dev = opt.rng;
  p.b0 = opt.b0;
  p.h0 = opt.h0;
  p.H_total = opt.H_total;
  p.bias = opt.bias;
  p.dbias = opt.dbias;
  p.h_major = (opt.bias.data != nullptr && opt.bias.sB == 0 && B > 1) ? 1 : 0;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.Sq_ctr = static_cast<int>(Sq);
  p.Sk_ctr = static_cast<int>(Sk);
  p.drop_bits = dropout_p > 0.0 ? opt.bits : nullptr;
  p.bits_kw = round_up(Sk, 128) / 32;
  p.bits_rows = round_up(Sq, 128);
  p.D_io = static_cast<int>(D);
  p.dk_io = strided(dk);
  p.dv_io = strided(dv);
  p.k_io = strided(k);
  p.acc_w = static_cast<int>(Da < 128 ? Da : 128);
  p.dq_acc = dq_acc;
  p.dq_part = opt.det ? dq_region : nullptr;
  p.part_stride = static_cast<size_t>(slice);
  p.lse2 = lse2;
  p.delta = delta;
  p.err = err;
  p.wait_limit_ns = wait_limit_ns();
  if (opt.dbias.data != nullptr && is_causal) {
    // key tiles above the diagonal are never visited: their dbias is 0
    e = launch_dbias_zero_causal(opt.dbias, static_cast<int>(B), static_cast<int>(H),
                                 static_cast<int>(Sq), static_cast<int>(Sk), stream);
    if (e != cudaSuccess) return SDPA_ERR_CUDA;
  }
  e = record_event(opt.ev_begin, stream);
  if (e == cudaSuccess)
    e = launch_bwd_main(static_cast<int>(Dk), is_causal != 0, dropout_p > 0.0, maps, p, stream);
  if (e == cudaSuccess) e = record_event(opt.ev_end, stream);
  if (e != cudaSuccess) return SDPA_ERR_CUDA;

  if (opt.det) {
    SumParams sp;
    sp.B = pp.B;
    sp.H = pp.H;
    sp.Sq = pp.Sq;
    sp.Sq_pad = pp.Sq_pad;
    sp.D = pp.D;
    sp.D_io = pp.D_io;
    sp.n_kv_tiles = p.n_kv_tiles;
    sp.causal = is_causal != 0;
    sp.scale = scale;
    sp.dq_part = dq_region;
    sp.cu_q = cu_q;
    sp.cu_k = cu_k;
    sp.part_stride = static_cast<size_t>(slice);
    sp.dq = strided(dq);
    return finish(launch_bwd_dq_sum(sp, stream), stream);
  }
  ConvParams cp;
  cp.B = pp.B;
  cp.H = pp.H;
  cp.Sq = pp.Sq;
  cp.Sq_pad = pp.Sq_pad;
  cp.D = pp.D;
  cp.D_io = pp.D_io;
  cp.scale = scale;
  cp.dq_acc = dq_acc;
  cp.cu_q = cu_q;
  cp.dq = strided(dq);
  return finish(launch_bwd_dq_convert(cp, stream), stream);
}

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" {

sdpa_status sdpa_fwd_ex(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                        double dropout_p, int is_causal, float scale, uint64_t seed,
                        uint64_t offset, sdpa_tensor* out, float* lse,
                        const sdpa_options* options, sdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  sdpa_status s = check_dims(q, k, v);
  if (s != SDPA_OK) return s;
  if ((s = check_common(dropout_p, scale)) != SDPA_OK) return s;
  const int64_t B = q->size[0], H = q->size[1], Sq = q->size[2], Sk = k->size[2], D = q->size[3];
  if (!head_dim_supported(D)) return SDPA_ERR_UNSUPPORTED;
  if ((s = check_tensor(q, B, H, Sq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(k, B, H, Sk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(v, B, H, Sk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(out, B, H, Sq, D)) != SDPA_OK) return s;
  if (D > 128 && options && options->attn_bias) return SDPA_ERR_UNSUPPORTED;
  if (B * H * Sq == 0) return SDPA_OK;
  if (Sk == 0) return SDPA_ERR_INVALID_ARG;  // softmax over no keys
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return SDPA_ERR_INVALID_ARG;
  Opts opt;
  if ((s = resolve_options(options, B, H, Sq, Sk, &opt)) != SDPA_OK) return s;
  if ((s = check_bits(opt, D, dropout_p, false)) != SDPA_OK) return s;
  return fwd_launch(q, k, v, out, lse, B, H, Sq, Sk, D, dropout_p, is_causal, scale, seed, offset,
                    opt, nullptr, nullptr, 0, stream);
}

sdpa_status sdpa_fwd_varlen(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                            const sdpa_varlen* seqs, double dropout_p, int is_causal, float scale,
                            uint64_t seed, uint64_t offset, sdpa_tensor* out, float* lse,
                            const sdpa_options* options, sdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  sdpa_status s = check_dims(q, k, v);
  if (s != SDPA_OK) return s;
  if ((s = check_common(dropout_p, scale)) != SDPA_OK) return s;
  const int64_t H = q->size[1], Tq = q->size[2], Tk = k->size[2], D = q->size[3];
  if ((s = check_varlen(seqs, q, k)) != SDPA_OK) return s;
  if (!head_dim_supported(D)) return SDPA_ERR_UNSUPPORTED;
  if ((s = check_tensor(q, 1, H, Tq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(k, 1, H, Tk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(v, 1, H, Tk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(out, 1, H, Tq, D)) != SDPA_OK) return s;
  if (H * Tq == 0) return SDPA_OK;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return SDPA_ERR_INVALID_ARG;
  if (options && (options->attn_bias || options->dbias)) return SDPA_ERR_UNSUPPORTED;
  const int64_t B = seqs->batch, Mq = seqs->max_seqlen_q, Mk = seqs->max_seqlen_k;
  Opts opt;
  if ((s = resolve_options(options, B, H, Mq, Mk, &opt)) != SDPA_OK) return s;
  if ((s = check_bits(opt, D, dropout_p, true)) != SDPA_OK) return s;
  return fwd_launch(q, k, v, out, lse, B, H, Mq, Mk, D, dropout_p, is_causal, scale, seed, offset,
                    opt, seqs->cu_seqlens_q, seqs->cu_seqlens_k, Tq, stream);
}

sdpa_status sdpa_fwd(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                     double dropout_p, int is_causal, float scale, uint64_t seed,
                     uint64_t offset, sdpa_tensor* out, float* lse, sdpa_stream_t stream) {
  return sdpa_fwd_ex(q, k, v, dropout_p, is_causal, scale, seed, offset, out, lse, nullptr,
                     stream);
}

size_t sdpa_bwd_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D) {
  (void)Sk;
  if (B <= 0 || H <= 0 || Sq <= 0 || D <= 0) return 0;
  return checked_bytes(B, H, round_up(Sq, 128), dq_acc_width(D) + 2);
}

size_t sdpa_dropout_bits_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk) {
  if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0) return 0;
  // B*H*ceil128(Sq)*ceil128(Sk)/8 bytes = B*H*ceil128(Sq) rows of ceil128(Sk)/32 words
  const double bytes = static_cast<double>(B) * static_cast<double>(H) *
                       static_cast<double>(round_up(Sq, 128)) * static_cast<double>(round_up(Sk, 128)) / 8.0;
  if (bytes > 4.0e18) return SIZE_MAX;
  return static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(round_up(Sq, 128)) *
         static_cast<size_t>(round_up(Sk, 128) / 32) * 4u;
}

size_t sdpa_bwd_workspace_size_ex(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D,
                                  const sdpa_options* options) {
  if (!options || !options->deterministic) return sdpa_bwd_workspace_size(B, H, Sq, Sk, D);
  if (B <= 0 || H <= 0 || Sq <= 0 || D <= 0 || Sk <= 0) return 0;
  return checked_bytes(B, H, round_up(Sq, 128), dq_acc_width(D) * ((Sk + 127) / 128) + 2);
}

sdpa_status sdpa_bwd_ex(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                        const sdpa_tensor* v, const sdpa_tensor* out, const float* lse,
                        double dropout_p, int is_causal, uint64_t seed, uint64_t offset,
                        float scale, sdpa_tensor* dq, sdpa_tensor* dk, sdpa_tensor* dv,
                        void* workspace, size_t workspace_bytes, const sdpa_options* options,
                        sdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  sdpa_status s = check_dims(q, k, v);
  if (s != SDPA_OK) return s;
  if ((s = check_common(dropout_p, scale)) != SDPA_OK) return s;
  const int64_t B = q->size[0], H = q->size[1], Sq = q->size[2], Sk = k->size[2], D = q->size[3];
  if (!head_dim_supported(D)) return SDPA_ERR_UNSUPPORTED;
  if (D > 128 && options && (options->attn_bias || options->dbias)) return SDPA_ERR_UNSUPPORTED;
  if ((s = check_tensor(q, B, H, Sq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(k, B, H, Sk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(v, B, H, Sk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dout, B, H, Sq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(out, B, H, Sq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dq, B, H, Sq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dk, B, H, Sk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dv, B, H, Sk, D)) != SDPA_OK) return s;
  if (B * H == 0) return SDPA_OK;
  if (Sq == 0) {
    // no queries: the key and value gradients are zero
    cudaError_t e = launch_zero_fill(strided(dk), B, H, Sk, D, stream);
    if (e == cudaSuccess) e = launch_zero_fill(strided(dv), B, H, Sk, D, stream);
    return finish(e, stream);
  }
  if (Sk == 0) return SDPA_ERR_INVALID_ARG;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return SDPA_ERR_INVALID_ARG;
  Opts opt;
  if ((s = resolve_options(options, B, H, Sq, Sk, &opt)) != SDPA_OK) return s;
  if ((s = check_bits(opt, D, dropout_p, false)) != SDPA_OK) return s;
  return bwd_launch(dout, q, k, v, out, lse, B, H, Sq, Sk, D, dropout_p, is_causal, seed, offset,
                    scale, dq, dk, dv, workspace, workspace_bytes, options, opt, nullptr, nullptr, 0,
                    stream);
}

sdpa_status sdpa_bwd(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                     const sdpa_tensor* v, const sdpa_tensor* out, const float* lse,
                     double dropout_p, int is_causal, uint64_t seed, uint64_t offset,
                     float scale, sdpa_tensor* dq, sdpa_tensor* dk, sdpa_tensor* dv,
                     void* workspace, size_t workspace_bytes, sdpa_stream_t stream) {
  return sdpa_bwd_ex(dout, q, k, v, out, lse, dropout_p, is_causal, seed, offset, scale, dq, dk,
                     dv, workspace, workspace_bytes, nullptr, stream);
}

size_t sdpa_bwd_varlen_workspace_size(const sdpa_varlen* seqs, int64_t H, int64_t D,
                                      const sdpa_options* options) {
  if (!seqs) return 0;
  return sdpa_bwd_workspace_size_ex(seqs->batch, H, seqs->max_seqlen_q, seqs->max_seqlen_k, D,
                                    options);
}

sdpa_status sdpa_bwd_varlen(const sdpa_tensor* dout, const sdpa_tensor* q, const sdpa_tensor* k,
                            const sdpa_tensor* v, const sdpa_tensor* out, const float* lse,
                            const sdpa_varlen* seqs, double dropout_p, int is_causal,
                            uint64_t seed, uint64_t offset, float scale, sdpa_tensor* dq,
                            sdpa_tensor* dk, sdpa_tensor* dv, void* workspace,
                            size_t workspace_bytes, const sdpa_options* options,
                            sdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  sdpa_status s = check_dims(q, k, v);
  if (s != SDPA_OK) return s;
  if ((s = check_common(dropout_p, scale)) != SDPA_OK) return s;
  const int64_t H = q->size[1], Tq = q->size[2], Tk = k->size[2], D = q->size[3];
  if ((s = check_varlen(seqs, q, k)) != SDPA_OK) return s;
  if (!head_dim_supported(D)) return SDPA_ERR_UNSUPPORTED;
  if ((s = check_tensor(q, 1, H, Tq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(k, 1, H, Tk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(v, 1, H, Tk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dout, 1, H, Tq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(out, 1, H, Tq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dq, 1, H, Tq, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dk, 1, H, Tk, D)) != SDPA_OK) return s;
  if ((s = check_tensor(dv, 1, H, Tk, D)) != SDPA_OK) return s;
  if (H == 0 || Tk == 0) return SDPA_OK;  // no keys: nothing to write
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return SDPA_ERR_INVALID_ARG;
  if (options && (options->attn_bias || options->dbias)) return SDPA_ERR_UNSUPPORTED;
  const int64_t B = seqs->batch, Mq = seqs->max_seqlen_q, Mk = seqs->max_seqlen_k;
  Opts opt;
  if ((s = resolve_options(options, B, H, Mq, Mk, &opt)) != SDPA_OK) return s;
  if ((s = check_bits(opt, D, dropout_p, true)) != SDPA_OK) return s;
  return bwd_launch(dout, q, k, v, out, lse, B, H, Mq, Mk, D, dropout_p, is_causal, seed, offset,
                    scale, dq, dk, dv, workspace, workspace_bytes, options, opt,
                    seqs->cu_seqlens_q, seqs->cu_seqlens_k, Tq, stream);
}

sdpa_status sdpa_dropout_mask_debug_ex(int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                       double dropout_p, uint64_t seed, uint64_t offset,
                                       const sdpa_options* options, uint8_t* mask,
                                       sdpa_stream_t stream_) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0) return SDPA_ERR_INVALID_ARG;
  if (!(dropout_p >= 0.0 && dropout_p < 1.0)) return SDPA_ERR_INVALID_ARG;
  const int64_t total = B * H * Sq * Sk;
  if (total == 0) return SDPA_OK;
  if (!mask) return SDPA_ERR_INVALID_ARG;
  if (H > 0x7fffffff) return SDPA_ERR_INVALID_ARG;
  Opts opt;
  const sdpa_status s = resolve_options(options, B, H, Sq, Sk, &opt);
  if (s != SDPA_OK) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int64_t blocks = (total + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks > 152 * 32 ? 152 * 32 : blocks);
  dropout_mask_kernel<<<grid, 256, 0, stream>>>(total, Sq * Sk, static_cast<int>(H), opt.b0,
                                                opt.h0, opt.H_total, drop_threshold(dropout_p),
                                                philox_key(seed, offset), opt.rng, mask);
  return finish(cudaGetLastError(), stream);
}

sdpa_status sdpa_dropout_mask_debug(int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                    double dropout_p, uint64_t seed, uint64_t offset,
                                    uint8_t* mask, sdpa_stream_t stream) {
  return sdpa_dropout_mask_debug_ex(B, H, Sq, Sk, dropout_p, seed, offset, nullptr, mask, stream);
}

sdpa_status sdpa_check_device(sdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SDPA_ERR_CUDA;
  uint32_t* err = error_word();
  if (!err) return SDPA_ERR_CUDA;
  uint32_t host = 0;
  if (cudaMemcpy(&host, err, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SDPA_ERR_CUDA;
  if (host != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return SDPA_ERR_CUDA;
    return SDPA_ERR_DEVICE_TIMEOUT;
  }
  return SDPA_OK;
}

sdpa_status sdpa_selftest_wait_timeout(uint64_t limit_ns, sdpa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint32_t* err = error_word();
  if (!err) return SDPA_ERR_CUDA;
  if (limit_ns == 0 || limit_ns > 10ull * 1000 * 1000 * 1000) return SDPA_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  if (cudaGetLastError() != cudaSuccess) return SDPA_ERR_CUDA;
  return sdpa_check_device(stream_);
}

const char* sdpa_status_string(sdpa_status status) {
  switch (status) {
    case SDPA_OK: return "SDPA_OK";
    case SDPA_ERR_INVALID_ARG: return "SDPA_ERR_INVALID_ARG: invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "SDPA_ERR_UNSUPPORTED: unsupported shape, layout or option (D a multiple of 8 in [8, 256], innermost; no attention bias above D = 128 or with a packed batch)";
    case SDPA_ERR_ALIGNMENT: return "SDPA_ERR_ALIGNMENT: base pointers and strides must be 16-byte aligned";
    case SDPA_ERR_CUDA: return "SDPA_ERR_CUDA: CUDA launch or driver call failed";
    case SDPA_ERR_DEVICE_TIMEOUT: return "SDPA_ERR_DEVICE_TIMEOUT: a kernel gave up on a bounded wait";
    case SDPA_ERR_WORKSPACE: return "SDPA_ERR_WORKSPACE: workspace missing, misaligned or too small";
  }
  return "SDPA_ERR_UNKNOWN";
}

}  // extern "C"
