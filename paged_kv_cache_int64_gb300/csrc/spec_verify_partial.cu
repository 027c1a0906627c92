// spec_verify_partial.cu - pkv_spec_verify_attn_partial: speculative-decode verify attention over
// an int8 per-token-head KV cache, as split-KV partials.
//
// HyperQwen PR #91 (_spec_attn_partial in spec_decode_attn.py): each request verifies T draft
// tokens against its long cached prefix; K/V are read through blk = table[req][pos // BLOCK_SIZE]
// with the block id widened to int64, and the int8 per-token-head scales are addressed with the
// same block id; the key range is cut into splits whose partials are merged by log-sum-exp.
//
// sm_103a design, one CTA = (split, KV head, request, token group), launched longest first (see
// the launch order below); the tokens x g query heads that share the KV head form N = 32 query
// columns (floor(32 / g) tokens per CTA: with T * g > 32 the tokens are spread over adjacent CTAs
// that read the same keys, or go to the N = 48 shape when that needs fewer CTAs; columns past the
// CTA's tokens are zero padding, so a T = 1 decode step runs on the same kernel), and the MMAs are
// "swapped" so the 128 keys of a tile are the M dimension (the verify step is HBM-bound at ~63 flop
// per cache byte):
//   warps 0, 3 TMA producers (K and V): Q once; per 128-key tile, the int8 (or e4m3) codes of K
//              (warp 0) and of V (warp 3) through 4-D maps over the paged pool (block id as a
//              coordinate), each into its own two-stage ring: 2 copies for a tile inside one
//              block, per-segment copies (gcd(block_size, 128) keys) across blocks.
//   warp 1     QK issuer: S^T = K Q^T (tcgen05.mma kind::f16, M=128 keys, N=32, K=256; K read
//              from tensor memory, Q fp16 in shared memory; S^T double-buffered in tensor memory).
//   warp 2     (after allocating tensor memory) PV issuer: O^T += V^T P^T (two M=128 halves of
//              head_dim, N=32, K=128 keys; V MN-major fp16 and P^T fp16 in shared memory). Two
//              issuing threads, because a tile's 32 small MMAs take longer to issue than to run.
//   warps 8-11 K converter: thread k owns key row k and widens it into the tile's tensor-memory K
//              buffer (two buffers, so tile j+1 is widened while tile j is scored), then releases
//              the K stage.
//   warps 12-15, 20-23 V converter, one warpgroup per head_dim half: once the previous PV has read
//              its half of the V tile, thread k widens its half of V row k into it (shared memory,
//              MN-major) and releases the V stage. No stage waits for the
//              softmax, and the K side keeps running while the V side waits for PV. int8 -> fp16
//              by byte permute (fp16 bits 0x6400|(b^0x80) equal 1024 + b + 128, so one
//              subtraction of 1152 gives b exactly - the int8->fp16 method of Kim et al. 2022,
//              "Who Says Elephants Can't Run"); e4m3 -> fp16 by the hardware conversion (exact;
//              the per-tensor scales multiply the scores and the output).
//   warps 4-7, 16-19, 24-27, 28-31 softmax, four warpgroups of 8 query columns each: thread k owns
//              key k's 8 scores of its group (TMEM lane k of S^T) and reads the key's K and V
//              scales from the scale pools itself, two tiles ahead; scores scaled by the K scale;
//              column maxima by a shuffle reduce-scatter per warp and shared memory across the
//              group's four warps, after which lane l keeps column (l & 7)'s running max (moved
//              only when it grows by more than 2^8) and broadcasts it by shuffles; P^T = p * v_scale
//              in fp16 into one of two buffers, so the softmax waits for the PV two tiles back (and
//              for the last one only to rescale O^T); the stored weights reduced per tile to column
//              sums that lane l keeps for column (l & 7); at the end, normalised partial O and its
//              LSE. (The 48-column shape: three groups of 16 columns, see Geo.)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <queue>
#include <utility>
#include <vector>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kD = 256;
constexpr int kBN = 128;  // keys per tile
constexpr int kChunk8 = 128 * 128;      // int8 [128 rows][128 B] swizzled chunk
constexpr int kChunk16 = 128 * 128;     // fp16 [128 rows][64] swizzled chunk
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_k(int st) { return st ? 128u : 0u; }    // 2 x 128: fp16 K rows
constexpr float kRescaleThreshold = 8.0f;
constexpr int kOrderMaxReqs = 128;  // batches up to this many requests run longest-first
constexpr int kStageCodes = 0;                   // a K or V stage: [2 chunks][128 rows][128 B] codes
constexpr int kStageBytes = 2 * kChunk8;         // 32 KB

// Two CTA shapes. N = 32 query columns: four softmax groups of 8 columns, 1,024 threads, K and V
// code rings of two stages each. N = 48 (e.g. 8 tokens x 6 heads): three groups of 16 columns,
// 896 threads, a single V code stage, so that the larger Q and P^T tiles fit in shared memory.
// Shared memory (1024-aligned): Q [4 chunks][N rows][128 B], the K code ring, the V code ring (K
// and V rings apart, so the K codes of tile j+2 can stream in as soon as tile j's K is widened,
// without waiting for its V), the fp16 V tile, two P^T buffers. P^T is MN-major: a key's N fp16
// weights are one row of 64 B (N = 32, 64-byte swizzle) or 128 B (N = 48 in a 64-column atom,
// 128-byte swizzle). Tensor memory: K 2 x 128 columns, S^T 2 x N, O^T 2 halves x N.
template <int kCols>
struct Geo {
  static_assert(kCols == 32 || kCols == 48, "two CTA shapes");
  static constexpr int kNQ = kCols;                      // query columns (tokens x group)
  static constexpr int kGC = kCols == 32 ? 8 : 16;       // query columns per softmax group
  static constexpr int kGroups = kNQ / kGC;              // 4 or 3 softmax warpgroups
  static constexpr int kThreads = kCols == 32 ? 1024 : 896;
  static constexpr int kVStages = kCols == 32 ? 2 : 1;
  static constexpr int kQChunk = kNQ * 128;              // fp16 [N rows][64] swizzled chunk
  static constexpr int kPRow = kCols == 32 ? 64 : 128;   // bytes per key row of P^T
  static constexpr int kPBuf = kBN * kPRow;              // one P^T buffer (a tile's 128 keys)
  static constexpr uint32_t kPLayout = kCols == 32 ? kLayoutSW64 : kLayoutSW128;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKStage = kOffQ + 4 * kQChunk;
  static constexpr int kOffVStage = kOffKStage + 2 * kStageBytes;
  static constexpr int kOffV16 = kOffVStage + kVStages * kStageBytes;
  static constexpr int kOffP = kOffV16 + 4 * kChunk16;
  static constexpr int kTiles = kOffP + 2 * kPBuf;
  __host__ __device__ static constexpr uint32_t col_s(int st) { return 256u + (uint32_t)(st * kNQ); }
  static constexpr uint32_t kColO = 256u + 2u * kNQ;     // O^T halves (head_dim 0-127, 128-255)
  static_assert(kOffKStage % 1024 == 0 && kOffV16 % 1024 == 0 && kOffP % 1024 == 0, "1024-B atoms");
  static_assert(kColO + 2 * kNQ <= kTmemCols, "tensor memory");
};

template <int kCols>
struct alignas(16) Barriers {
  uint64_t q_full, q_ready;
  uint64_t kst_full[2], kst_free[2];  // K stage ring (freed by the K converter)
  uint64_t vst_full[2], vst_free[2];  // V stage ring (freed by the V converter)
  uint64_t k_ready[2], k_free[2];     // K_j in TMEM buffer j%2; QK_j done with it
  uint64_t v_ready[2];                // half h (head_dim 128h..128h+127) of V_j widened into shared memory
  uint64_t v_free[2];                 // half h of the V tile read by PV_j
  uint64_t s_full[2];                 // S^T_j in TMEM buffer j%2
  uint64_t s_free[2];                 // S^T_j read by every softmax thread: QK_{j+2} may overwrite it
  uint64_t p_full[2];                 // P^T_j (buffer j%2) written, O^T rescaled; per tile parity,
                                      // since the softmax may run a tile ahead of the MMA's wait
  uint64_t pv_done[2];                // PV_j complete (V tile and P^T buffer j%2 free, O^T current),
                                      // one barrier per tile parity (the softmax waits two tiles back)
  uint64_t drain;                     // after a wait gave up: both issuers' MMAs are complete
  uint32_t armed[5];                  // TMA phases armed: q_full, kst_full[0..1], vst_full[0..1]
  uint32_t tmem_base;
  int abort;
  uint32_t kbad[2], vbad[2];        // per stage: segments whose block id was out of range
  float red[2][Geo<kCols>::kGroups][4][Geo<kCols>::kGC];  // [tile parity][group][warp][column]: maxima, then the final sums
  float inv_l[kCols];      // epilogue: 1 / column sum
};

struct Params {
  CUtensorMap qmap;   // bf16 [R*T][Hq][D]: dims {D, Hq, R*T}, box {64, g, T}
  CUtensorMap k8map;  // int8 pool: dims {D, Hkv, bs, nb}, box {128, 1, G, 1}
  CUtensorMap v8map;
  CUtensorMap k8map_big;  // box {128, 1, 128, 1}: a whole tile inside one block (bs >= 128)
  CUtensorMap v8map_big;
  int32_t big_ok;
  const int32_t* block_table;
  int64_t bt_stride, num_blocks;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t num_reqs;
  int32_t T, group, num_q_heads, block_size, seg, split_tokens, max_splits;
  int32_t tpc, n_tg;  // tokens per CTA (tpc * group <= 32 query columns) and CTAs per (split, head)
  float scale_log2;
  float* part_o;
  float* part_lse;
  int64_t rows;  // num_reqs * T * Hq
  int* dev_err;
  const float* k_descale;  // fp8 cache: per-tensor scales (device scalars)
  const float* v_descale;
  const float* k_scale;    // int8 cache: per-token-head scales [nb][bs][Hkv], read by the softmax
  const float* v_scale;
  int64_t scale_stride_blk, scale_stride_tok;
  uint64_t wait_limit_ns;  // bound on each wait (kWaitLimitNs unless a test shortens it)
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 16 int8 codes -> 16 fp16 integers, exact (byte-permute + one fp16 subtraction per pair).
__device__ __forceinline__ void widen16_f16(uint4 in, uint32_t (&o)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;
    uint32_t lo = __byte_perm(u, 0x64646464u, 0x5140);
    uint32_t hi = __byte_perm(u, 0x64646464u, 0x7362);
    __half2 hl = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
    __half2 hh = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
    o[2 * i] = *reinterpret_cast<uint32_t*>(&hl);
    o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&hh);
  }
}

// 16 e4m3 codes -> 16 fp16 values, exact (every e4m3 value is an fp16 value): hardware conversion.
__device__ __forceinline__ void widen16_e4m3(uint4 in, uint32_t (&o)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * i]) : "h"((uint16_t)(w[i] & 0xffffu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * i + 1]) : "h"((uint16_t)(w[i] >> 16)));
  }
}

template <bool kFp8>
__device__ __forceinline__ void widen16(uint4 in, uint32_t (&o)[8]) {
  if (kFp8) widen16_e4m3(in, o); else widen16_f16(in, o);
}

// Reduce-scatter of 16 columns: on entry every lane holds 16 column values; on exit every lane holds
// the warp maximum (kMax) or sum of column (lane & 15). 16 shuffles.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter8(float (&v)[8], int lane) {
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int q = 0; q < o; ++q) {
      const float keep = upper ? v[q + o] : v[q];
      const float send = upper ? v[q] : v[q + o];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[q] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  float x = v[0];
#pragma unroll
  for (int o = 8; o <= 16; o <<= 1) {
    const float other = __shfl_xor_sync(0xffffffffu, x, o);
    x = kMax ? fmaxf(x, other) : x + other;
  }
  return x;
}
template <bool kMax>
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int q = 0; q < o; ++q) {
      const float keep = upper ? v[q + o] : v[q];
      const float send = upper ? v[q] : v[q + o];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[q] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  const float other = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return kMax ? fmaxf(v[0], other) : v[0] + other;
}

// Column maxima of 16 columns without consuming the input (the scores are needed afterwards): the
// first exchange (lanes 8 apart) writes 8 partial maxima to a scratch array, the rest runs on that.
__device__ __forceinline__ float reduce_scatter16_max_keep(const float (&v)[16], int lane) {
  float t[8];
  const bool upper = (lane & 8) != 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float keep = upper ? v[q + 8] : v[q];
    const float send = upper ? v[q] : v[q + 8];
    t[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int q = 0; q < o; ++q) {
      const float keep = up ? t[q + o] : t[q];
      const float send = up ? t[q] : t[q + o];
      t[q] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  return fmaxf(t[0], __shfl_xor_sync(0xffffffffu, t[0], 16));
}

template <int kGC, bool kMax>
__device__ __forceinline__ float reduce_scatter(float (&v)[kGC], int lane) {
  if constexpr (kGC == 8) return reduce_scatter8<kMax>(v, lane);
  else return reduce_scatter16<kMax>(v, lane);
}
template <int kGC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[kGC]) {
  if constexpr (kGC == 8) tmem_ld_32x32b_x8(taddr, r);
  else tmem_ld_32x32b_x16(taddr, r);
}
template <int kGC>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[kGC]) {
  if constexpr (kGC == 8) tmem_st_32x32b_x8(taddr, r);
  else tmem_st_32x32b_x16(taddr, r);
}

template <bool kFp8, int kCols>
__global__ void __launch_bounds__(Geo<kCols>::kThreads, 1) spec_verify_partial_kernel(const __grid_constant__ Params p) {
  using Gm = Geo<kCols>;
  constexpr int kNQ = Gm::kNQ, kGC = Gm::kGC, kGroups = Gm::kGroups, kVStages = Gm::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Gm::kOffQ;
  uint8_t* sV16 = smem + Gm::kOffV16;
  uint8_t* sP = smem + Gm::kOffP;
  Barriers<kCols>& bar = *reinterpret_cast<Barriers<kCols>*>(smem + Gm::kTiles);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The linear CTA index is (request, split) pair * (KV heads * token groups) + KV head * token
  // groups + token group: the CTAs that share a key range are adjacent, so they run together and
  // the later reads of the same K/V tiles hit L2.
  const int64_t lin = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
  const int units = (int)gridDim.y * p.n_tg;
  const int64_t pair = lin / units;
  const int kvh = (int)(lin - pair * units) / p.n_tg;
  const int t_base = ((int)(lin - pair * units) - kvh * p.n_tg) * p.tpc;  // first query token of this CTA
  const int nq = min(p.tpc, p.T - t_base) * p.group;                     // live query columns; the rest pad
  int r, split;
  if (p.num_reqs <= kOrderMaxReqs) {
    // Longest first: the CTAs run in launch order, one per SM, so the pairs with a whole
    // split_tokens keys go first (request by request) and the requests' shorter last splits
    // follow from the longest down; the short CTAs then fill in behind the long ones instead of
    // trailing them. Pairs past the last one have nothing to do and leave after one barrier.
    int* s_rest = reinterpret_cast<int*>(sP);  // scratch before any role starts (P^T buffers)
    long long* s_wsum = reinterpret_cast<long long*>(s_rest + kOrderMaxReqs);
    int* s_pick = reinterpret_cast<int*>(s_wsum + kOrderMaxReqs / 32);
    const int t = threadIdx.x;
    int n_full = 0, rest = 0;
    if (t < p.num_reqs) {
      const int len = max(__ldg(p.seq_lens + t), 0);
      n_full = min(len / p.split_tokens, p.max_splits);
      rest = n_full < p.max_splits ? len - n_full * p.split_tokens : 0;  // keys of the last, shorter split
    }
    long long inc = n_full;  // inclusive prefix sum of the whole-split counts over requests 0..t
    if (t < kOrderMaxReqs) {
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) s_wsum[warp] = inc;
      s_rest[t] = rest;
    }
    if (t == 0) s_pick[0] = s_pick[1] = -1;
    const int n_short = __syncthreads_count(rest > 0);
    long long n_full_pairs = 0;
#pragma unroll
    for (int w = 0; w < kOrderMaxReqs / 32; ++w) {
      if (w < warp) inc += s_wsum[w];
      n_full_pairs += s_wsum[w];
    }
    if (pair >= n_full_pairs + n_short) return;  // CTA-uniform: no pair this far down the order
    if (t < p.num_reqs) {
      if (pair < n_full_pairs) {
        if (pair >= inc - n_full && pair < inc) {
          s_pick[0] = t;
          s_pick[1] = (int)(pair - (inc - n_full));
        }
      } else if (rest > 0) {
        int rank = 0;  // shorter last splits ranked by length, longest first (ties: lower request)
        for (int u = 0; u < p.num_reqs; ++u) rank += s_rest[u] > rest || (s_rest[u] == rest && u < t);
        if (rank == pair - n_full_pairs) {
          s_pick[0] = t;
          s_pick[1] = n_full;
        }
      }
    }
    __syncthreads();
    r = s_pick[0];
    split = s_pick[1];
    // the scratch is overwritten only after the CTA-wide barrier that follows the tensor-memory
    // allocation, by which time every thread has read its pick
  } else {
    r = (int)(pair / p.max_splits);
    split = (int)(pair - (int64_t)r * p.max_splits);
  }
  const int seq_len = __ldg(p.seq_lens + r);
  const int64_t k_begin64 = (int64_t)split * p.split_tokens;
  if (k_begin64 >= seq_len) return;  // CTA-uniform: split past this request's keys
  const int k_begin = (int)k_begin64;
  const int k_end = min(seq_len, k_begin + p.split_tokens);
  const int n_tiles = (k_end - k_begin + kBN - 1) / kBN;
  const int prefix = seq_len - p.T;  // query token t sits at position prefix + t

  if (threadIdx.x == 0) {
    // the last launched split must reach seq_len; keys past max_splits * split_tokens are lost
    const bool short_grid = split == p.max_splits - 1 && (int64_t)k_begin + p.split_tokens < seq_len;
    if (short_grid || prefix < 0) record_error(p.dev_err, kErrDeviceBounds);
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_ready, 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar.kst_full[s], 1);
      mbar_init(&bar.kst_free[s], 128);
      mbar_init(&bar.vst_full[s], 1);
      mbar_init(&bar.vst_free[s], 256);
      mbar_init(&bar.k_ready[s], 128);
      mbar_init(&bar.k_free[s], 1);
      mbar_init(&bar.s_full[s], 1);
      mbar_init(&bar.s_free[s], kGroups * 128);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bar.v_ready[h], 128);
      mbar_init(&bar.v_free[h], 1);
    }
    mbar_init(&bar.p_full[0], kGroups * 128);  // every softmax thread of every group
    mbar_init(&bar.p_full[1], kGroups * 128);
    mbar_init(&bar.pv_done[0], 1);
    mbar_init(&bar.pv_done[1], 1);
    mbar_init(&bar.drain, 2);  // the QK and the PV issuer
    for (int b = 0; b < 5; ++b) bar.armed[b] = 0;
    bar.abort = 0;
    fence_mbar_init();
  }
  if (prefix < 0) return;  // CTA-uniform (after the error is noted)
  if (warp == 2) {
    tmem_alloc(&bar.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  volatile int* abort = &bar.abort;
  const uint64_t wl = p.wait_limit_ns;
  const int G = p.seg;

  if (warp == 0 || warp == 3) {
    // ---------------------------------------------------------------------------- producers
    // warp 0 streams the K codes, warp 3 the V codes, each through its own ring (K: two stages; V:
    // two, or one with N = 48); both read the block table for their tiles
    const bool is_k = warp == 0;
    const int nst = is_k ? 2 : kVStages;
    const int nseg = kBN / G;
    if (is_k && lane == 0) {
      mbar_arm_tx(&bar.q_full, 4u * 128u * (uint32_t)(p.tpc * p.group), &bar.armed[0]);  // the whole box
      for (int c = 0; c < 4; ++c)
        tma_load_3d(sQ + c * Gm::kQChunk, &p.qmap, &bar.q_full, c * 64, kvh * p.group, r * p.T + t_base);
    }
    uint64_t* full = is_k ? bar.kst_full : bar.vst_full;
    uint64_t* freeb = is_k ? bar.kst_free : bar.vst_free;
    uint32_t* badw = is_k ? bar.kbad : bar.vbad;
    uint32_t* armed = bar.armed + (is_k ? 1 : 3);
    const CUtensorMap* codes = is_k ? &p.k8map : &p.v8map;
    const CUtensorMap* codes_big = is_k ? &p.k8map_big : &p.v8map_big;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = nst == 2 ? (j & 1) : 0;
      const int round = nst == 2 ? (j >> 1) : j;  // uses of this stage before tile j
      uint8_t* stage = smem + (is_k ? Gm::kOffKStage : Gm::kOffVStage) + st * kStageBytes;
      // go / stop is lane 0's wait result, broadcast, so the lanes never part (once any role gives
      // up, every wait returns false promptly)
      bool ok0 = true;
      if (lane == 0 && round >= 1) ok0 = mbar_wait_suspend(&freeb[st], (round - 1) & 1, abort, wl);
      if (!__shfl_sync(0xffffffffu, ok0, 0)) break;
      const int key0 = k_begin + j * kBN;
      int blk = -1;
      if (lane < nseg && key0 + lane * G < k_end) {
        const int pos = key0 + lane * G;
        const int col = pos / p.block_size;
        blk = col < p.max_blocks ? __ldg(p.block_table + (int64_t)r * p.bt_stride + col) : -2;
        if (blk < 0 || (int64_t)blk >= p.num_blocks) blk = -2;
      }
      const uint32_t bad = __ballot_sync(0xffffffffu, blk == -2);
      const uint32_t nloaded = __popc(__ballot_sync(0xffffffffu, blk >= 0));
      const int blk0 = __shfl_sync(0xffffffffu, blk, 0);
      const int slot0 = key0 % p.block_size;
      // the 128 keys lie in one valid block: 2 copies of 128 rows
      const bool big = p.big_ok && bad == 0 && blk0 >= 0 && slot0 + kBN <= p.block_size;
      if (lane == 0) {
        if (bad) record_error(p.dev_err, kErrDeviceBounds);
        badw[st] = bad;
        const uint32_t rows = big ? (uint32_t)kBN : nloaded * (uint32_t)G;
        mbar_arm_tx(&full[st], rows * 2u * 128u, &armed[st]);  // the copies below always follow
        if (big)
          for (int c = 0; c < 2; ++c)
            tma_load_4d(stage + kStageCodes + c * kChunk8, codes_big, &full[st], c * 128, kvh, slot0, blk0);
      }
      __syncwarp();
      if (!big && blk >= 0) {
        const int slot = (key0 + lane * G) % p.block_size;
        for (int c = 0; c < 2; ++c)
          tma_load_4d(stage + kStageCodes + c * kChunk8 + lane * G * 128, codes, &full[st], c * 128, kvh, slot, blk);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------------------- QK issuer
    // S^T_j = K_j Q^T into TMEM buffer j%2, once K_j is in TMEM and every softmax thread has read
    // S^T_{j-2} out of that buffer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_f16(128, kNQ, false, false, false);
      const uint32_t q_base = smem_u32(sQ);
      bool ok = mbar_wait_suspend(&bar.q_ready, 0, abort, wl);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait_suspend(&bar.s_free[st], ((j - 2) >> 1) & 1, abort, wl)) break;
        if (!mbar_wait_suspend(&bar.k_ready[st], (j >> 1) & 1, abort, wl)) break;
        tc_fence_after();
        for (int ks = 0; ks < 16; ++ks)
          umma_f16_ts(tmem + Gm::col_s(st), tmem + col_k(st) + ks * 8,
                      smem_desc(q_base + (ks >> 2) * Gm::kQChunk + (ks & 3) * 32, 16, 1024), id_qk, ks > 0);
        umma_commit(&bar.s_full[st]);
        umma_commit(&bar.k_free[st]);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---------------------------------------------------------------------------- PV issuer
    // O^T += V_j^T P^T_j, each head_dim half as soon as its V half is widened; a second issuing
    // thread, so the 16 QK and 16 PV MMAs of a tile are issued side by side
    if (lane == 0) {
      constexpr uint32_t id_pv = idesc_f16(128, kNQ, false, true, true);
      const uint32_t v_base = smem_u32(sV16), p_base = smem_u32(sP);
      for (int i = 0; i < n_tiles; ++i) {
        if (!mbar_wait_suspend(&bar.p_full[i & 1], (i >> 1) & 1, abort, wl)) break;
        const uint32_t pb = p_base + (i & 1) * Gm::kPBuf;
        bool ok = true;
        for (int hh = 0; hh < 2 && ok; ++hh) {
          if (!mbar_wait_suspend(&bar.v_ready[hh], i & 1, abort, wl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int ks = 0; ks < 8; ++ks)
            umma_f16_ss(tmem + Gm::kColO + hh * kNQ, smem_desc(v_base + hh * 2 * kChunk16 + ks * 2048, kChunk16, 1024),
                        smem_desc(pb + ks * 16 * Gm::kPRow, 0, 8 * Gm::kPRow, Gm::kPLayout), id_pv,
                        (i > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bar.v_free[hh]);
        }
        if (!ok) break;
        umma_commit(&bar.pv_done[i & 1]);
      }
    }
    __syncwarp();
  } else if (warp >= 8 && warp < 12) {
    // ---------------------------------------------------------------------------- K converter
    // thread k owns key row k of each tile: its int8 (or e4m3) K row -> fp16 into TMEM lane k of the
    // tile's K buffer. A row outside the split or in a bad block holds stale stage bytes: int8 codes
    // widen to finite values whatever they are, and such a key's score is masked (past the split)
    // or multiplied by a zero scale (bad block), so the row is widened as it is; e4m3 rows are
    // zeroed first, since a stale NaN code would survive the mask as 0 * NaN in the MMA. First, Q
    // bf16 -> fp16 in place (N rows x 256).
    const int quarter = warp & 3;
    const int k = quarter * 32 + lane;
    const int kseg = k / G;  // the key's segment within a tile (bad-block bits)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    bool dead = !__all_sync(0xffffffffu, mbar_wait_suspend(&bar.q_full, 0, abort, wl));
    if (!dead) {  // (row, chunk) pairs idx = k, k + 128, ...; padding rows (past the CTA's columns) become zeros
      for (int idx = k; idx < 4 * kNQ; idx += 128) {
        const int row = idx % kNQ, c = idx / kNQ;
        const bool live_row = row < nq;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4* ptr = reinterpret_cast<uint4*>(sQ + c * Gm::kQChunk + row * 128 + q * 16);
          uint4 v = live_row ? *ptr : make_uint4(0, 0, 0, 0);
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            w[e] = pack_f16x2(f.x, f.y);
          }
          *ptr = v;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar.q_ready);
    }
    for (int j = 0; j < n_tiles && !dead; ++j) {
      const int st = j & 1;
      const uint8_t* kstage = smem + Gm::kOffKStage + st * kStageBytes;
      bool got = mbar_wait_suspend(&bar.kst_full[st], (j >> 1) & 1, abort, wl);
      if (got && j >= 2) got = mbar_wait_suspend(&bar.k_free[st], ((j >> 1) - 1) & 1, abort, wl);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const bool live = k_begin + j * kBN + k < k_end && !((bar.kbad[st] >> kseg) & 1u);
#pragma unroll 1
      for (int w8 = 0; w8 < 8; ++w8) {  // 32 codes = 16 TMEM columns per step
        uint32_t kv[16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int q8 = 2 * (w8 & 3) + i;
          const uint4 v = *reinterpret_cast<const uint4*>(kstage + kStageCodes + (w8 >> 2) * kChunk8 + k * 128 +
                                                          ((q8 ^ (k & 7)) * 16));
          uint32_t o[8];
          widen16<kFp8>((kFp8 && !live) ? make_uint4(0, 0, 0, 0) : v, o);  // zero codes widen to zeros
#pragma unroll
          for (int e = 0; e < 8; ++e) kv[8 * i + e] = o[e];
        }
        tmem_st_32x32b_x16(tmem + lane_off + col_k(st) + 16 * w8, kv);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar.k_ready[st]);
      mbar_arrive(&bar.kst_free[st]);
    }
  } else if ((warp >= 12 && warp < 16) || (warp >= 20 && warp < 24)) {
    // ---------------------------------------------------------------------------- V converter
    // two warpgroups, one per half of head_dim (warps 12-15: 0-127, warps 20-23: 128-255), each with
    // its own ready / free barriers, so half 0 of V_{j+1} is widened while PV_j still reads half 1.
    // Thread k owns key row k: its half V row -> fp16 into the MN-major V tile. A row outside the
    // split or in a bad block meets a zero P^T entry: int8 rows are widened as they are (finite
    // whatever the stale bytes), e4m3 rows are zeroed first (0 * NaN would not vanish).
    const int hv = warp >= 20 ? 1 : 0;  // warps 20-23: the second half
    const int k = (warp & 3) * 32 + lane;
    const int kseg = k / G;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = kVStages == 2 ? (j & 1) : 0;
      const int round = kVStages == 2 ? (j >> 1) : j;  // uses of this stage before tile j
      const uint8_t* vstage = smem + Gm::kOffVStage + st * kStageBytes;
      bool got = j == 0 || mbar_wait_suspend(&bar.v_free[hv], (j - 1) & 1, abort, wl);
      if (got) got = mbar_wait_suspend(&bar.vst_full[st], round & 1, abort, wl);
      if (!__all_sync(0xffffffffu, got)) break;
      const bool live = k_begin + j * kBN + k < k_end && !((bar.vbad[st] >> kseg) & 1u);
      const uint8_t* src = vstage + kStageCodes + hv * kChunk8 + k * 128;
      uint8_t* dst = sV16 + 2 * hv * kChunk16 + k * 128;
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        uint4 v = *reinterpret_cast<const uint4*>(src + ((q8 ^ (k & 7)) * 16));
        if (kFp8 && !live) v = make_uint4(0, 0, 0, 0);
        uint32_t o[8];
        widen16<kFp8>(v, o);
        uint8_t* row = dst + (q8 >> 2) * kChunk16;
        const uint32_t piece = 2u * (q8 & 3);
        *reinterpret_cast<uint4*>(row + ((piece ^ (k & 7)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(row + (((piece + 1) ^ (k & 7)) * 16)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar.v_ready[hv]);
      mbar_arrive(&bar.vst_free[st]);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------------------- softmax
    // warpgroups of kGC query columns (N = 32: four groups of 8, warps 4-7, 16-19, 24-27, 28-31;
    // N = 48: three groups of 16, warps 4-7, 16-19, 24-27); thread k holds key k's kGC scores of
    // its group (TMEM lane k of S^T). Column maxima: a shuffle reduce-scatter leaves column
    // (lane % kGC)'s warp maximum in the lane, shared memory combines the group's four warps; lane l
    // then keeps column (l % kGC)'s running max (the same in all four warps) and hands it to the
    // other lanes by shuffles. The K scale folds into the scores, the V scale into P^T; each
    // thread reads its key's two scales from the cache itself, two tiles ahead (the block id three
    // tiles ahead), so no stage buffer waits for the softmax and the HBM latency is covered.
    const int grp = warp < 8 ? 0 : warp < 20 ? 1 : warp < 28 ? 2 : 3;
    const int c0 = kGC * grp;      // the group's first query column
    const int cl = lane & (kGC - 1);  // this lane keeps the running max of column c0 + cl
    const int quarter = warp & 3;
    const int k = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float k_descale = kFp8 ? __ldg(p.k_descale) : 0.0f;
    // block id of this thread's key in tile jj (-1: past the split or a bad table entry)
    // Position of this thread's key in the pool, advanced tile by tile without divisions:
    // (col, slot) of key k_begin + t * 128 + k, for the tile t whose block id is looked up next.
    const int q128 = kBN / p.block_size, r128 = kBN % p.block_size;
    int col_t = (k_begin + k) / p.block_size, slot_t = (k_begin + k) % p.block_size;
    auto advance = [&]() {
      col_t += q128;
      slot_t += r128;
      if (slot_t >= p.block_size) {
        slot_t -= p.block_size;
        ++col_t;
      }
    };
    // block id of the key in tile jj (at the current (col_t, slot_t)); -1 past the split or bad
    auto key_block = [&](int jj) -> int {
      if (k_begin + jj * kBN + k >= k_end || col_t >= p.max_blocks) return -1;
      const int blk = __ldg(p.block_table + (int64_t)r * p.bt_stride + col_t);
      return (blk < 0 || (int64_t)blk >= p.num_blocks) ? -1 : blk;
    };
    // the key's K and V scales in a tile with block id blk and slot slot (0 for a dead key: its K
    // and V rows are zero)
    auto key_scales = [&](int blk, int slot, float& ks, float& vs) {
      ks = vs = 0.0f;
      if (blk >= 0) {
        const int64_t off = (int64_t)blk * p.scale_stride_blk + (int64_t)slot * p.scale_stride_tok + kvh;
        ks = __ldg(p.k_scale + off);
        vs = __ldg(p.v_scale + off);
      }
    };
    // scales of tiles j and j+1, block id and slot of tile j+2 (e4m3: per-tensor scales on scores
    // and output)
    float ks_cur = 0.0f, vs_cur = 1.0f, ks_1 = 0.0f, vs_1 = 1.0f;
    int blk_2 = -1, slot_2 = 0;
    if (!kFp8) {
      key_scales(key_block(0), slot_t, ks_cur, vs_cur);
      advance();
      key_scales(key_block(1), slot_t, ks_1, vs_1);
      advance();
      blk_2 = key_block(2);
      slot_2 = slot_t;
    }
    // column sums: each tile's weights are reduced across the warp once they are stored, and lane l
    // keeps the running sum of column c0 + (l % kGC) (no per-key partial sums in registers)
    float l_col = 0.0f;
    float m_col = -INFINITY;
    bool dead = false;  // warp-uniform; the named barrier below is reached the same number of times
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j & 1;
      const int key0 = k_begin + j * kBN;
      const int key = key0 + k;
      const bool in_range = key < k_end;
      // tile j+2's scales and tile j+3's block id are fetched while this tile is scored
      float ks_2 = 0.0f, vs_2 = 1.0f;
      if (!kFp8) {
        key_scales(blk_2, slot_2, ks_2, vs_2);
        advance();
        blk_2 = key_block(j + 3);
        slot_2 = slot_t;
      }
      if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait_suspend(&bar.s_full[st], (j >> 1) & 1, abort, wl));
      float s[kGC];
      {
        uint32_t v[kGC];
        const float ks = kFp8 ? k_descale : ks_cur;
        if (!dead) {
          tc_fence_after();
          tmem_ld_cols<kGC>(tmem + lane_off + Gm::col_s(st) + c0, v);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bar.s_free[st]);  // QK_{j+2} may now overwrite this S^T buffer
        }
        const float f = p.scale_log2 * ks;
        if (!dead && key0 + kBN <= k_end && c0 + kGC <= nq && key0 + kBN - 1 <= prefix) {
#pragma unroll
          for (int q = 0; q < kGC; ++q) s[q] = __uint_as_float(v[q]) * f;
        } else if (key0 + kBN - 1 <= prefix) {  // every key of the tile precedes the first draft token
#pragma unroll
          for (int q = 0; q < kGC; ++q)
            s[q] = (!dead && in_range && c0 + q < nq) ? __uint_as_float(v[q]) * f : -INFINITY;
        } else {  // causal limit of column c (token t_base + c / group): key <= prefix + that token
#pragma unroll
          for (int q = 0; q < kGC; ++q) {
            const int c = c0 + q;
            const bool vis = !dead && in_range && c < nq && key <= prefix + t_base + c / p.group;
            s[q] = vis ? __uint_as_float(v[q]) * f : -INFINITY;
          }
        }
      }
      {
        float mine;
        if constexpr (kGC == 16) {
          mine = reduce_scatter16_max_keep(s, lane);
        } else {
          float t[kGC];
#pragma unroll
          for (int q = 0; q < kGC; ++q) t[q] = s[q];
          mine = reduce_scatter<kGC, true>(t, lane);
        }
        if (lane < kGC) bar.red[st][grp][quarter][lane] = mine;
      }
      named_bar_sync(1 + grp, 128);
      // column c0 + cl: tile maximum, running maximum and rescale factor
      const float cmax = fmaxf(fmaxf(bar.red[st][grp][0][cl], bar.red[st][grp][1][cl]),
                               fmaxf(bar.red[st][grp][2][cl], bar.red[st][grp][3][cl]));
      float alpha = 1.0f;
      bool rescale = false;
      if (m_col == -INFINITY || cmax > m_col + kRescaleThreshold) {
        const float m_new = fmaxf(m_col, cmax);
        if (m_new != -INFINITY) {
          rescale = m_col != -INFINITY;
          alpha = rescale ? ex2_approx(m_col - m_new) : 0.0f;
          m_col = m_new;
        }
      }
      const float mu = m_col == -INFINITY ? 0.0f : m_col;
      const bool any_rescale = __any_sync(0xffffffffu, rescale);  // the same in all four warps
      // P^T buffer j%2 was last read by PV_{j-2}; O^T may be rescaled only once PV_{j-1} is done
      if (!dead && j >= 2)
        dead = !__all_sync(0xffffffffu, mbar_wait_suspend(&bar.pv_done[j & 1], ((j - 2) >> 1) & 1, abort, wl));
      if (!dead && any_rescale && j >= 1)
        dead = !__all_sync(0xffffffffu, mbar_wait_suspend(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, wl));
      // P = exp2(s - m): the column maxima are broadcast from their lanes first, then the exps and
      // the fp16 P^T stores run as independent batches
      // (16 columns: in place over the scores, which keeps the registers within the 896-thread budget)
      float e_buf[kGC == 16 ? 1 : kGC];
      float (&e)[kGC] = *reinterpret_cast<float(*)[kGC]>(kGC == 16 ? s : e_buf);
      if constexpr (kGC == 16) {
#pragma unroll
        for (int q = 0; q < kGC; ++q) e[q] = ex2_approx(s[q] - __shfl_sync(0xffffffffu, mu, q));
      } else {
#pragma unroll
        for (int q = 0; q < kGC; ++q) e[q] = __shfl_sync(0xffffffffu, mu, q);
#pragma unroll
        for (int q = 0; q < kGC; ++q) e[q] = ex2_approx(s[q] - e[q]);
      }
      if (!dead) {  // P^T for key k (columns c0 .. c0 + kGC - 1 of buffer j % 2): p * v_scale, fp16
        const float vs = vs_cur;
        // row k of the MN-major P^T, the group's 16-byte chunks; the swizzle XORs a chunk index with
        // the row's bits at 128-byte granularity (64-B rows: bits 1-2 of k; 128-B rows: bits 0-2)
        uint8_t* prow = sP + (j & 1) * Gm::kPBuf + k * Gm::kPRow;
        const uint32_t sw = Gm::kPRow == 64 ? ((uint32_t)(k >> 1) & 3u) : ((uint32_t)k & 7u);
#pragma unroll
        for (int cc = 0; cc < kGC / 8; ++cc) {
          uint32_t h[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __half2 t = __floats2half2_rn(e[8 * cc + 2 * q] * vs, e[8 * cc + 2 * q + 1] * vs);
            h[q] = *reinterpret_cast<const uint32_t*>(&t);
          }
          const uint32_t chunk = (uint32_t)(grp * (kGC / 8) + cc);
          *reinterpret_cast<uint4*>(prow + ((chunk ^ sw) * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
      {  // the weights are stored: reduce them (in place) to the tile's column sums
        const float tsum = reduce_scatter<kGC, false>(e, lane);
        l_col = (rescale ? l_col * alpha : l_col) + tsum;  // column c0 + cl, with its own factor
      }
      if (!dead) {
        tc_fence_after();
        if (any_rescale) {  // O^T lane k (head_dim index) times column c0 + q's factor
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[kGC];
            tmem_ld_cols<kGC>(tmem + lane_off + Gm::kColO + hh * kNQ + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < kGC; ++q)
              v[q] = __float_as_uint(__uint_as_float(v[q]) * __shfl_sync(0xffffffffu, alpha, q));
            tmem_st_cols<kGC>(tmem + lane_off + Gm::kColO + hh * kNQ + c0, v);
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar.p_full[j & 1]);
      }
      ks_cur = ks_1;
      vs_cur = vs_1;
      ks_1 = ks_2;
      vs_1 = vs_2;
    }
    // epilogue: column sums, O^T / l, log-sum-exp (each group for its kGC columns)
    bool fin = !dead && !*abort && mbar_wait_suspend(&bar.pv_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, abort, wl);
    fin = __all_sync(0xffffffffu, fin);
    named_bar_sync(1 + grp, 128);  // every warp of the group is past its last read of bar.red
    {
      if (lane < kGC) bar.red[0][grp][quarter][lane] = l_col;
    }
    named_bar_sync(1 + grp, 128);
    if (quarter == 0 && lane < kGC) {  // lane q: column c0 + q's sum, 1 / l and log-sum-exp
      const int c = c0 + lane;
      const float l = bar.red[0][grp][0][lane] + bar.red[0][grp][1][lane] + bar.red[0][grp][2][lane] +
                      bar.red[0][grp][3][lane];
      // e4m3: the per-tensor V scale multiplies the output once
      bar.inv_l[c] = l > 0.0f ? (kFp8 ? __ldg(p.v_descale) / l : 1.0f / l) : 0.0f;
      if (fin && c < nq) {
        const int t = t_base + c / p.group, hh = c % p.group;
        const int64_t row = ((int64_t)r * p.T + t) * p.num_q_heads + (int64_t)kvh * p.group + hh;
        p.part_lse[(int64_t)split * p.rows + row] = l > 0.0f ? (m_col + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
    named_bar_sync(1 + grp, 128);
    if (fin) {
      tc_fence_after();
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t v[kGC];
        tmem_ld_cols<kGC>(tmem + lane_off + Gm::kColO + hh * kNQ + c0, v);
        tmem_wait_ld();
        const int d = hh * 128 + k;
#pragma unroll
        for (int q = 0; q < kGC; ++q) {
          const int c = c0 + q;
          if (c >= nq) break;
          const int t = t_base + c / p.group, h2 = c % p.group;
          const int64_t row = ((int64_t)r * p.T + t) * p.num_q_heads + (int64_t)kvh * p.group + h2;
          p.part_o[((int64_t)split * p.rows + row) * kD + d] = __uint_as_float(v[q]) * bar.inv_l[c];
        }
      }
    }
  }

  tc_fence_before();
  // every role has left its loop; the flag's final value, the same for every thread (a thread that
  // set it reads it set, so the OR over the CTA sees it)
  const bool gave_up = __syncthreads_or(*abort != 0);
  if (gave_up) {
    // some wait gave up: before the tensor memory is freed and the CTA exits, wait for what this
    // CTA still has in flight - the TMA copies of every phase it armed and every MMA it issued
    if ((warp == 0 || warp == 3) && lane == 0) {
      if (warp == 0) drain_armed(&bar.q_full, bar.armed[0]);
      const int b = warp == 0 ? 1 : 3;
      drain_armed(warp == 0 ? &bar.kst_full[0] : &bar.vst_full[0], bar.armed[b]);
      drain_armed(warp == 0 ? &bar.kst_full[1] : &bar.vst_full[1], bar.armed[b + 1]);
    }
    if ((warp == 1 || warp == 2) && lane == 0) {
      umma_commit(&bar.drain);  // arrives once every MMA this thread issued is complete
      mbar_wait_drain(&bar.drain, 0);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && gave_up) record_error(p.dev_err, kErrTimeout);
}

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

}  // namespace

}  // namespace pkv

extern "C" size_t pkv_spec_verify_workspace_bytes(int32_t num_tokens, int32_t num_q_heads, int32_t head_dim,
                                                  int32_t max_splits) {
  if (num_tokens <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_splits <= 0) return 0;
  const size_t rows = (size_t)num_tokens * (size_t)num_q_heads * (size_t)max_splits;
  const size_t o = (rows * (size_t)head_dim * 4 + 255) & ~(size_t)255;
  const size_t l = (rows * 4 + 255) & ~(size_t)255;
  return o + l;
}

namespace pkv {
namespace {

template <bool kFp8, int kCols>
void launch_shape(const Params& p, dim3 grid, cudaStream_t st) {
  constexpr int kSmem = 1024 + Geo<kCols>::kTiles + (int)sizeof(Barriers<kCols>);
  static_assert(kSmem <= 227 * 1024, "dynamic shared memory of one CTA");
  static std::atomic<uint64_t> attr_done{0};
  once_per_device(attr_done, [] {
    cudaFuncSetAttribute(spec_verify_partial_kernel<kFp8, kCols>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  spec_verify_partial_kernel<kFp8, kCols><<<grid, Geo<kCols>::kThreads, kSmem, st>>>(p);
}

// Shared host path of the int8 (per-token-head scales) and fp8 (per-tensor descales) verify calls.
template <bool kFp8>
pkv_status launch_verify(const char* name, const void* q, const void* k_cache, const void* v_cache,
                         const float* k_sc, const float* v_sc, int64_t num_blocks, int64_t stride_blk,
                         int64_t stride_tok, int64_t stride_head, int64_t scale_stride_blk,
                         int64_t scale_stride_tok, const int32_t* block_table, int64_t bt_stride,
                         int32_t max_blocks, const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         float softmax_scale, int32_t split_tokens, int32_t max_splits, float* part_o,
                         float* part_lse, int32_t* dev_err, void* stream) {
  clear_error();
  PKV_UNSUP(head_dim == kD, "%s: head_dim must be 256 (got %d)", name, head_dim);
  if (num_reqs == 0) return PKV_OK;  // nothing to do, nothing read
  PKV_ARG(q && k_cache && v_cache && k_sc && v_sc && block_table && seq_lens && part_o && part_lse,
          "%s: null pointer argument", name);
  PKV_ARG(num_reqs > 0 && T > 0 && num_q_heads > 0 && num_kv_heads > 0 && num_blocks > 0 && block_size > 0 &&
              max_blocks > 0 && bt_stride >= max_blocks && max_splits > 0 && split_tokens > 0,
          "%s: bad size argument", name);
  PKV_UNSUP(num_q_heads % num_kv_heads == 0, "%s: num_q_heads %% num_kv_heads != 0", name);
  const int group = num_q_heads / num_kv_heads;
  PKV_UNSUP(group <= 32, "%s: num_q_heads / num_kv_heads must be at most 32 (got %d)", name, group);
  // CTA shape: N = 48 query columns when that serves a key range with fewer CTAs than N = 32
  // (e.g. 8 tokens x 6 heads in one CTA instead of two), else N = 32
  const int tpc32 = T < 32 / group ? T : 32 / group, n32 = (T + tpc32 - 1) / tpc32;
  const int tpc48 = T < 48 / group ? T : 48 / group, n48 = (T + tpc48 - 1) / tpc48;
  const bool wide = n48 < n32;
  const int tpc = wide ? tpc48 : tpc32;  // tokens per CTA
  const int n_tg = wide ? n48 : n32;     // CTAs per (split, KV head, request)
  PKV_ARG((int64_t)max_splits * n_tg < (1ll << 31), "%s: grid too large", name);
  PKV_UNSUP(block_size % 8 == 0, "%s: block_size must be a multiple of 8", name);
  PKV_UNSUP(split_tokens % kBN == 0, "%s: split_tokens must be a multiple of 128", name);
  PKV_ARG(stride_blk > 0 && stride_tok > 0 && stride_head > 0 && (kFp8 || (scale_stride_blk > 0 && scale_stride_tok > 0)),
          "%s: strides must be positive", name);
  PKV_ARG(aligned16(q) && aligned16(k_cache) && aligned16(v_cache) && stride_blk % 16 == 0 && stride_tok % 16 == 0 &&
              stride_head % 16 == 0,
          "%s: q, caches and cache strides must be 16-byte aligned", name);
  PKV_ARG(kFp8 || ((reinterpret_cast<uintptr_t>(k_sc) & 3) == 0 && (reinterpret_cast<uintptr_t>(v_sc) & 3) == 0 &&
                   scale_stride_tok >= num_kv_heads),
          "%s: scale pools must be 4-byte aligned, with scale_stride_tok >= num_kv_heads", name);
  PKV_ARG(softmax_scale > 0.0f, "%s: softmax_scale must be positive", name);
  Params p{};
  const int G = gcd_int(block_size, kBN);
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)num_q_heads, (uint64_t)num_reqs * (uint64_t)T};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)num_q_heads * kD * 2};
    const uint32_t box[3] = {64, (uint32_t)group, (uint32_t)tpc};
    pkv_status s = encode_tiled(&p.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, "q");
    if (s != PKV_OK) return s;
  }
  {
    const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)num_kv_heads, (uint64_t)block_size, (uint64_t)num_blocks};
    const uint64_t strides[3] = {(uint64_t)stride_head, (uint64_t)stride_tok, (uint64_t)stride_blk};
    const uint32_t box[4] = {128, 1, (uint32_t)G, 1};
    pkv_status s = encode_tiled(&p.k8map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, k_cache, dims, strides, box, "k_cache");
    if (s != PKV_OK) return s;
    s = encode_tiled(&p.v8map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, v_cache, dims, strides, box, "v_cache");
    if (s != PKV_OK) return s;
    p.big_ok = block_size >= kBN;
    if (p.big_ok) {
      const uint32_t big[4] = {128, 1, (uint32_t)kBN, 1};
      s = encode_tiled(&p.k8map_big, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, k_cache, dims, strides, big, "k_cache");
      if (s != PKV_OK) return s;
      s = encode_tiled(&p.v8map_big, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, v_cache, dims, strides, big, "v_cache");
      if (s != PKV_OK) return s;
    }
  }
  if (!kFp8) {
    p.k_scale = k_sc;
    p.v_scale = v_sc;
    p.scale_stride_blk = scale_stride_blk;
    p.scale_stride_tok = scale_stride_tok;
  } else {
    p.k_descale = k_sc;
    p.v_descale = v_sc;
  }
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks;
  p.seq_lens = seq_lens;
  p.num_reqs = num_reqs;
  p.T = T;
  p.group = group;
  p.tpc = tpc;
  p.n_tg = n_tg;
  p.num_q_heads = num_q_heads;
  p.block_size = block_size;
  p.seg = G;
  p.split_tokens = split_tokens;
  p.max_splits = max_splits;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.rows = (int64_t)num_reqs * T * num_q_heads;
  p.dev_err = dev_err;
  p.wait_limit_ns = take_wait_limit_ns();
  dim3 grid((unsigned)(max_splits * n_tg), (unsigned)num_kv_heads, (unsigned)num_reqs);
  if (wide)
    launch_shape<kFp8, 48>(p, grid, static_cast<cudaStream_t>(stream));
  else
    launch_shape<kFp8, 32>(p, grid, static_cast<cudaStream_t>(stream));
  return check_launch(name);
}

}  // namespace
}  // namespace pkv

// Host-side planning: the launch's CTAs run longest first, one per SM, so the kernel time is about
// the makespan of a longest-processing-time-first list schedule of its CTAs: every (split, KV head,
// token group) CTA costs kCtaUs plus kTileUs per 128-key tile (x1.4 for the 48-column shape), and
// every CTA past a request's keys kEmptyUs (constants fitted to GB300 timings of a 32-request batch
// swept over ten split sizes, residual 2 us). The whole splits are all alike and go first, so they
// are dealt round-robin in closed form; the shorter last splits are placed greedily, longest first
// (beyond 8 per SM, where the greedy schedule is all but level, the makespan is taken as the mean
// load plus the largest of them, which keeps the planner linear in the batch); the empty CTAs then
// fill the idle time below the makespan before they extend it.
extern "C" int32_t pkv_spec_verify_pick_split(const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                              int32_t num_q_heads, int32_t num_kv_heads, int32_t num_sms) {
  using namespace pkv;
  if (!seq_lens || num_reqs <= 0 || T <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_sms <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  const int group = num_q_heads / num_kv_heads;
  if (group > 32) return 0;
  const int tpc32 = T < 32 / group ? T : 32 / group, n32 = (T + tpc32 - 1) / tpc32;
  const int tpc48 = T < 48 / group ? T : 48 / group, n48 = (T + tpc48 - 1) / tpc48;
  const bool wide = n48 < n32;
  const int64_t units = (int64_t)num_kv_heads * (wide ? n48 : n32);  // CTAs per (request, split)
  constexpr double kCtaUs = 7.5, kTileUs = 2.08, kEmptyUs = 2.0;
  const double tile_us = wide ? 1.4 * kTileUs : kTileUs;
  int64_t max_len = 0;
  for (int r = 0; r < num_reqs; ++r) max_len = std::max<int64_t>(max_len, std::max(seq_lens[r], 0));
  if (max_len == 0) return 1024;
  std::vector<int64_t> rests;
  std::vector<double> sm(num_sms);
  int32_t best_split = 0;
  double best = 0.0;
  for (int32_t split = 1024; split <= 16384; split += 512) {
    const int64_t ms = (max_len + split - 1) / split;
    int64_t n_full = 0;
    rests.clear();
    for (int r = 0; r < num_reqs; ++r) {
      const int64_t len = std::max(seq_lens[r], 0);
      n_full += len / split;
      if (len % split) rests.push_back(len % split);
    }
    // whole splits: F CTAs of equal cost dealt round-robin
    const int64_t F = n_full * units;
    const double full_us = kCtaUs + tile_us * (split / kBN);
    for (int i = 0; i < num_sms; ++i) sm[i] = (double)(F / num_sms + (i < F % num_sms ? 1 : 0)) * full_us;
    double makespan = 0.0, total = 0.0;
    if ((int64_t)rests.size() * units <= 8 * (int64_t)num_sms) {
      std::sort(rests.begin(), rests.end(), [](int64_t a, int64_t b) { return a > b; });
      std::priority_queue<std::pair<double, int>, std::vector<std::pair<double, int>>,
                          std::greater<std::pair<double, int>>> pq;
      for (int i = 0; i < num_sms; ++i) pq.push({sm[i], i});
      for (const int64_t rest : rests)
        for (int64_t u = 0; u < units; ++u) {
          auto top = pq.top();
          pq.pop();
          top.first += kCtaUs + tile_us * (double)((rest + kBN - 1) / kBN);
          pq.push(top);
        }
      while (!pq.empty()) {
        makespan = std::max(makespan, pq.top().first);
        total += pq.top().first;
        pq.pop();
      }
    } else {
      for (int i = 0; i < num_sms; ++i) {
        total += sm[i];
        makespan = std::max(makespan, sm[i]);
      }
      double largest = 0.0;
      for (const int64_t rest : rests) {
        const double d = kCtaUs + tile_us * (double)((rest + kBN - 1) / kBN);
        total += d * (double)units;
        largest = std::max(largest, d);
      }
      makespan = std::max(makespan, total / num_sms + largest);
    }
    // empty CTAs: first into the idle time below the makespan, the rest spread over every SM
    const int64_t empties = (int64_t)num_reqs * ms * units - (n_full + (int64_t)rests.size()) * units;
    const double idle = makespan * num_sms - total, extra = empties * kEmptyUs - idle;
    if (extra > 0.0) makespan += extra / num_sms;
    if (best_split == 0 || makespan < best) {
      best = makespan;
      best_split = split;
    }
  }
  return best_split;
}

extern "C" pkv_status pkv_spec_verify_attn_partial(const void* q, const int8_t* k_cache, const int8_t* v_cache,
                                                   const float* k_scale, const float* v_scale, int64_t num_blocks,
                                                   int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                                   int64_t scale_stride_blk, int64_t scale_stride_tok,
                                                   const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                                   const int32_t* seq_lens, int32_t num_reqs, int32_t T,
                                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                   int32_t block_size, float softmax_scale, int32_t split_tokens,
                                                   int32_t max_splits, float* part_o, float* part_lse,
                                                   int32_t* dev_err, void* stream) {
  return pkv::launch_verify<false>("spec_verify_attn_partial", q, k_cache, v_cache, k_scale, v_scale, num_blocks,
                                   stride_blk, stride_tok, stride_head, scale_stride_blk, scale_stride_tok,
                                   block_table, bt_stride, max_blocks, seq_lens, num_reqs, T, num_q_heads,
                                   num_kv_heads, head_dim, block_size, softmax_scale, split_tokens, max_splits,
                                   part_o, part_lse, dev_err, stream);
}

extern "C" pkv_status pkv_spec_verify_attn_partial_fp8(const void* q, const uint8_t* k_fp8, const uint8_t* v_fp8,
                                                       const float* k_descale, const float* v_descale,
                                                       int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                                                       int64_t stride_head, const int32_t* block_table,
                                                       int64_t bt_stride, int32_t max_blocks, const int32_t* seq_lens,
                                                       int32_t num_reqs, int32_t T, int32_t num_q_heads,
                                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                                       float softmax_scale, int32_t split_tokens, int32_t max_splits,
                                                       float* part_o, float* part_lse, int32_t* dev_err,
                                                       void* stream) {
  return pkv::launch_verify<true>("spec_verify_attn_partial_fp8", q, k_fp8, v_fp8, k_descale, v_descale, num_blocks,
                                  stride_blk, stride_tok, stride_head, 0, 0, block_table, bt_stride, max_blocks,
                                  seq_lens, num_reqs, T, num_q_heads, num_kv_heads, head_dim, block_size,
                                  softmax_scale, split_tokens, max_splits, part_o, part_lse, dev_err, stream);
}
