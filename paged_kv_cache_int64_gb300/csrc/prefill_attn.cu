// prefill_attn.cu - pkv_paged_prefill_attn: chunked causal prefill attention over a paged bf16
// KV cache, exact-QK (bf16) or int8-QK.
//
// HyperQwen PR #109 (_prefill_attn_kernel in prefill_attn_hd256.py; review: the "int8_qk=False"
// and "int8_qk=True" arms, chunk 2048, head_dim 256, block 880): for every query of the chunk,
// softmax(scale * q.K^T) V over the keys at or before its position, K and V read through the
// block table with the block id widened to int64 before the stride product.
//
// sm_103a design (one CTA = 128 query rows of one query head of one request):
//   warp 0      TMA producer: Q once; per 128-key tile, K and V gathered from the paged pool with
//               4-D tensor maps [head_dim, kv_heads, block_size, num_blocks] whose block
//               coordinate is the block id (the TMA unit forms the 64-bit address): a tile inside
//               one block is 4 copies of 128 rows per tensor; a tile across blocks is split into
//               segments of gcd(block_size, 128) keys, one lane per segment reading the table; the
//               next tile's block ids are read early.
//   warp 1      MMA issuer (one thread): S = Q K^T (tcgen05.mma kind::f16, M=128 N=128 K=256,
//               both operands in shared memory, f32 accumulator in tensor memory), then
//               O += P V (M=128 N=256 K=128) with P read from tensor memory and V MN-major.
//   warp 2      tensor-memory allocation (512 columns: O 256, S 128, two P buffers of 64). S is
//               single-buffered and released as soon as both softmax halves hold it in registers;
//               P (bf16 pairs) is double-buffered, so QK_{j+1} never waits for PV_{j-1}.
//   warps 4-11  softmax, two warpgroups that split every row (score columns 0-63 / 64-127, O
//               columns 0-127 / 128-255; row i lives in TMEM lane i): one tensor-memory read of S
//               per tile, scale, causal mask, row maximum shared through shared memory, running
//               max moved only when it grows by more than 2^8 (so O is rarely rescaled), exp2, P
//               packed to bf16 into its tensor-memory buffer, row sums of the rounded P; the
//               epilogue normalises O and stores bf16.
//   warps 12-15 int8-QK only: read the int8 K rows (dense scratch of kv_int8_stats_quant) and
//               widen them to fp16 integers in the K tile; half 0 of the softmax quantizes the Q
//               rows in place first. Q8.K8 runs as an f16 MMA: every product and partial sum is an
//               integer below 2^24, so the f32 accumulator holds the exact integer dot product.
// Rows of the last tile past seq_len (and of any out-of-range block) are zero-filled in shared
// memory before the MMAs read them, so stale or NaN pool bytes never reach P.V. Every wait is
// bounded: on expiry the CTA records PKV_ERR_TIMEOUT, drains and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "host_common.h"
#include "sm103.cuh"

namespace pkv {

namespace {

constexpr int kD = 256;
constexpr int kBM = 128;                // query rows per CTA
constexpr int kBN = 128;                // keys per tile
constexpr int kChunkBytes = 128 * 128;  // one [128 rows][64 x 16-bit] swizzled chunk
constexpr int kTileBytes = 4 * kChunkBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;   // S: 128 fp32 columns (one buffer)
constexpr uint32_t kColP0 = 384;  // P: two buffers of 64 columns (128 bf16 keys packed in pairs)
constexpr uint32_t kColP1 = 448;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// dynamic shared memory layout (1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kTilesEnd = kOffV + kTileBytes;

struct Barriers {
  uint64_t q_full;      // TMA Q landed
  uint64_t q_ready;     // int8: Q quantized in place
  uint64_t k_full[4];   // chunk c of K tile j ready (TMA bytes, or converter arrivals)
  uint64_t k_empty[4];  // chunk c of K tile j consumed by the QK MMAs
  uint64_t v_full;      // V tile j ready
  uint64_t fix;         // producer-private: copies of a tile that needs zero-filled rows
  uint64_t s_full;      // S_j in TMEM
  uint64_t s_free;      // S_j copied to registers by both softmax halves: QK_{j+1} may overwrite it
  // P_j / PV_j barriers, one per tile parity: the MMA issuer waits for P_{j-1} after QK_j and the
  // softmax for PV_{j-2}, so one barrier per kind could be two phases ahead of the phase waited
  // for, which a parity wait cannot tell apart from the phase itself
  uint64_t p_full[2];   // P_j in TMEM and O rescaled (256 softmax arrivals), tile parity j & 1
  uint64_t pv_done[2];  // PV_j complete (V free, O current), tile parity j & 1
  uint32_t tmem_base;
  int abort;
  float kscale[2][kBN];  // int8: per-key scales of the tile
  float qscale[kBM];     // int8: per-row q scales
  float rowmax[2][2][kBM];  // per tile parity, per half: row maxima (and the final row sums)
};

struct Params {
  CUtensorMap qmap;   // bf16 q: dims {D, Hq, total_q}, box {64, 1, 128}
  CUtensorMap kmap;   // bf16 pool: dims {D, Hkv, bs, nb}, box {64, 1, G, 1}
  CUtensorMap vmap;
  CUtensorMap kmap_big;  // same pool, box {64, 1, 128, 1}: a whole tile inside one block (bs >= 128)
  CUtensorMap vmap_big;
  int32_t big_ok;        // block_size >= 128
  const int8_t* k8;   // int8 scratch [R][max_ctx][Hkv][D] (read row by row by the converter)
  CUtensorMap k16map; // fp16 copy of the codes: dims {D, Hkv, R*max_ctx}, box {64, 1, 128}
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_blocks;
  int32_t max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t num_q_heads, group, block_size, seg;
  float scale_log2;
  const float* k8_scale;
  int64_t max_ctx;
  int32_t num_kv_heads;
  int32_t n_mtiles;
  __nv_bfloat16* out;
  int* dev_err;
  // fused fp8 (mode 3): the e4m3 pools, read row by row by the converter warps, and the
  // per-tensor scales (device scalars)
  const uint8_t* k_fp8;
  const uint8_t* v_fp8;
  int64_t stride_blk, stride_tok, stride_head;
  const float* k_scale;
  const float* v_scale;
};

// kMode 0: exact QK (bf16 K from the pool); 1: int8 QK with K widened from the int8 scratch by
// converter warps; 2: int8 QK with K read by TMA from the fp16 copy of the codes; 3: exact QK on a
// per-tensor e4m3 pool, K and V dequantized to bf16 tile by tile by converter warps.
template <int kMode>
struct Cfg {
  static constexpr int kThreads = (kMode == 1 || kMode == 3) ? 512 : 384;
  static constexpr int kTiles = kTilesEnd;
  static constexpr int kSmem = 1024 + kTiles + (int)sizeof(Barriers);
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Quantize this thread's Q row (row i of the swizzled bf16 Q tile) in place to fp16 integers and
// return its scale: absmax / 127 and codes rint(x * (127 / absmax)) clamped to +-127, the
// arithmetic of kv_int8_stats_quant.
__device__ float quantize_q_row_inplace(uint8_t* sQ, int i) {
  float amax = 0.0f;
  bool nan = false;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 v = *reinterpret_cast<const uint4*>(sQ + c * kChunkBytes + sw128_offset(i, q * 8));
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(b[e]);
        nan |= (f.x != f.x) | (f.y != f.y);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
  const bool live = !nan && amax > 0.0f;
  const float scale = nan ? __int_as_float(0x7fc00000) : (amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f);
  const float inv = live ? __fdiv_rn(127.0f, amax) : 0.0f;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint4* ptr = reinterpret_cast<uint4*>(sQ + c * kChunkBytes + sw128_offset(i, q * 8));
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        int c0 = 0, c1 = 0;
        if (live) {
          c0 = max(-127, min(127, __float2int_rn(__fmul_rn(f.x, inv))));
          c1 = max(-127, min(127, __float2int_rn(__fmul_rn(f.y, inv))));
        }
        const __half2 h = __halves2half2(__int2half_rn(c0), __int2half_rn(c1));
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *ptr = v;
    }
  }
  return scale;
}

// 16 int8 codes -> 16 fp16 integers (exact).
__device__ __forceinline__ void widen16(uint4 in, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b0 = (int)(int8_t)(w[i] & 0xffu), b1 = (int)(int8_t)((w[i] >> 8) & 0xffu);
    const int b2 = (int)(int8_t)((w[i] >> 16) & 0xffu), b3 = (int)(int8_t)(w[i] >> 24);
    const __half2 h01 = __halves2half2(__int2half_rn(b0), __int2half_rn(b1));
    const __half2 h23 = __halves2half2(__int2half_rn(b2), __int2half_rn(b3));
    o[2 * i] = *reinterpret_cast<const uint32_t*>(&h01);
    o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&h23);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Zero whole 128-byte rows (all four chunks) of a [4][128][128 B] tile: rows >= n_valid and rows
// of segments whose bit is set in bad_mask. Executed by one warp.
__device__ __forceinline__ void zero_rows(uint8_t* tile, int n_valid, uint32_t bad_mask, int G, int lane) {
  for (int idx = lane; idx < 4 * kBN * 8; idx += 32) {
    const int piece = idx & 7;
    const int row = (idx >> 3) & (kBN - 1);
    const int c = idx >> 10;
    if (row >= n_valid || ((bad_mask >> (row / G)) & 1u))
      *reinterpret_cast<uint4*>(tile + c * kChunkBytes + row * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
  }
}

template <int kMode>
__global__ void __launch_bounds__(Cfg<kMode>::kThreads, 1)
    paged_prefill_attn_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  Barriers& bar = *reinterpret_cast<Barriers*>(smem + Cfg<kMode>::kTiles);
  constexpr bool kInt8 = kMode == 1 || kMode == 2;  // int8 QK (quantized Q, per-key K scales, f16 MMA)
  constexpr bool kConv = kMode == 1;                 // K widened by the converter warps
  constexpr bool kFused = kMode == 3;                // K and V dequantized by the converter warps

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.z;
  const int qh = blockIdx.y;
  const int mt = p.n_mtiles - 1 - (int)blockIdx.x;  // latest (heaviest) tiles first
  const int kvh = qh / p.group;
  const int q0 = __ldg(p.qsl + r);
  const int q_len = __ldg(p.qsl + r + 1) - q0;
  const int seq_len = __ldg(p.seq_lens + r);
  if (mt * kBM >= q_len || q_len > seq_len) return;  // CTA-uniform
  const int rows_valid = min(kBM, q_len - mt * kBM);
  const int p0 = seq_len - q_len + mt * kBM;         // position of row 0
  const int kv_end = min(seq_len, p0 + rows_valid);  // keys [0, kv_end)
  const int n_tiles = (kv_end + kBN - 1) / kBN;
  const int tok0 = q0 + mt * kBM;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_ready, 128);
    for (int c = 0; c < 4; ++c) {
      mbar_init(&bar.k_full[c], (kConv || kFused) ? 128 : 1);
      mbar_init(&bar.k_empty[c], 1);
    }
    mbar_init(&bar.v_full, kFused ? 128 : 1);
    mbar_init(&bar.fix, 1);
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.s_free, 256);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar.p_full[b], 256);
      mbar_init(&bar.pv_done[b], 1);
    }
    bar.abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&bar.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  volatile int* abort = &bar.abort;

  if (warp == 0 && kFused) {
    // ---------------------------------------------------------------------------- producer (Q)
    if (lane == 0) {
      prefetch_tensormap(&p.qmap);
      mbar_arrive_expect_tx(&bar.q_full, kTileBytes);
      for (int c = 0; c < 4; ++c) tma_load_3d(sQ + c * kChunkBytes, &p.qmap, &bar.q_full, c * 64, qh, tok0);
    }
  } else if (warp == 0) {
    // ---------------------------------------------------------------------------- producer
    const int G = p.seg;
    const int nseg = kBN / G;
    const uint32_t seg_bytes = (uint32_t)G * 128u;  // one chunk of one segment
    if (lane == 0) {
      prefetch_tensormap(&p.qmap);
      prefetch_tensormap(&p.vmap);
      if (!kInt8) prefetch_tensormap(&p.kmap);
      if (kMode == 2) prefetch_tensormap(&p.k16map);
      if (p.big_ok) {
        prefetch_tensormap(&p.vmap_big);
        if (!kInt8) prefetch_tensormap(&p.kmap_big);
      }
      mbar_arrive_expect_tx(&bar.q_full, kTileBytes);
      for (int c = 0; c < 4; ++c) tma_load_3d(sQ + c * kChunkBytes, &p.qmap, &bar.q_full, c * 64, qh, tok0);
    }
    // block id of segment `lane` of tile j: >= 0, -1 past seq_len, -2 out-of-range entry
    auto lookup = [&](int j) -> int {
      const int pos = j * kBN + lane * G;
      if (lane >= nseg || pos >= seq_len) return -1;
      const int col = pos / p.block_size;
      if (col >= p.max_blocks) return -2;
      const int blk = __ldg(p.block_table + (int64_t)r * p.bt_stride + col);
      if (blk < 0 || (int64_t)blk >= p.num_blocks) return -2;
      return blk;
    };
    auto issue_seg = [&](uint8_t* tile, const CUtensorMap* map, uint64_t* mb, int blk, int key0) {
      const int slot = (key0 + lane * G) % p.block_size;
      for (int c = 0; c < 4; ++c) tma_load_4d(tile + c * kChunkBytes + lane * G * 128, map, mb, c * 64, kvh, slot, blk);
    };
    struct TileInfo {
      int blk;           // this lane's segment block id (>= 0), -1 past seq_len, -2 bad entry
      uint32_t bad;      // segments with a bad table entry
      uint32_t nloaded;  // segments with a valid block
      bool fix;          // rows to zero-fill: a tail past seq_len or a bad segment
      bool big;          // the 128 keys lie in one valid block: 4 copies of 128 rows per tensor
      int blk0, slot0;   // block and first slot of key 0 of the tile
    };
    auto info = [&](int j) -> TileInfo {
      TileInfo t;
      t.blk = j < n_tiles ? lookup(j) : -1;
      t.bad = __ballot_sync(0xffffffffu, t.blk == -2);
      t.nloaded = __popc(__ballot_sync(0xffffffffu, t.blk >= 0));
      t.fix = t.bad != 0 || seq_len - j * kBN < kBN;
      t.blk0 = __shfl_sync(0xffffffffu, t.blk, 0);
      t.slot0 = (j * kBN) % p.block_size;
      t.big = p.big_ok && t.bad == 0 && t.blk0 >= 0 && t.slot0 + kBN <= p.block_size;
      return t;
    };
    // a whole tile of one tensor with 4 copies of [128 rows][64 x 16-bit] (lane 0)
    auto issue_big = [&](uint8_t* tile, const CUtensorMap* map, uint64_t* mb, const TileInfo& t) {
      if (lane == 0)
        for (int c = 0; c < 4; ++c) tma_load_4d(tile + c * kChunkBytes, map, mb, c * 64, kvh, t.slot0, t.blk0);
    };
    uint32_t fix_phase = 0;
    // K tile j through k_full[c] (bf16) or the K8 stage (int8), chunk by chunk as QK_{j-1} frees it.
    // K rows past seq_len need no zero-fill (their scores are masked); rows of a bad segment do,
    // so such a tile goes through the private barrier, is patched, then published.
    auto load_k = [&](int j, const TileInfo& t) {
      const int key0 = j * kBN;
      if (kConv) return;  // the converter warps read the int8 K rows themselves
      if (kMode == 2) {   // fp16 copy of the int8 codes, dense by position: 4 copies of 128 rows
        if (lane == 0) {
          const int row = (int)((int64_t)r * p.max_ctx + key0);
          for (int c = 0; c < 4; ++c) {
            if (j > 0 && !mbar_wait(&bar.k_empty[c], (j - 1) & 1, abort)) break;
            mbar_arrive_expect_tx(&bar.k_full[c], (uint32_t)kChunkBytes);
            tma_load_3d(sK + c * kChunkBytes, &p.k16map, &bar.k_full[c], c * 64, kvh, row);
          }
        }
        __syncwarp();
        return;
      }
      if (t.bad) {
        if (lane == 0) {
          for (int c = 0; c < 4 && j > 0; ++c)
            if (!mbar_wait(&bar.k_empty[c], (j - 1) & 1, abort)) break;
          if (!*abort) mbar_arrive_expect_tx(&bar.fix, 4u * t.nloaded * seg_bytes);
        }
        __syncwarp();
        if (*abort) return;
        if (t.blk >= 0) issue_seg(sK, &p.kmap, &bar.fix, t.blk, key0);
        if (lane == 0) mbar_wait(&bar.fix, fix_phase & 1, abort);
        ++fix_phase;
        __syncwarp();
        if (*abort) return;
        zero_rows(sK, kBN, t.bad, G, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          for (int c = 0; c < 4; ++c) mbar_arrive(&bar.k_full[c]);
        __syncwarp();
        return;
      }
      if (t.big) {
        if (lane == 0) {
          for (int c = 0; c < 4; ++c) {
            if (j > 0 && !mbar_wait(&bar.k_empty[c], (j - 1) & 1, abort)) break;
            mbar_arrive_expect_tx(&bar.k_full[c], (uint32_t)kChunkBytes);
            tma_load_4d(sK + c * kChunkBytes, &p.kmap_big, &bar.k_full[c], c * 64, kvh, t.slot0, t.blk0);
          }
        }
        __syncwarp();
        return;
      }
      const int slot = (key0 + lane * G) % p.block_size;
      for (int c = 0; c < 4; ++c) {
        if (lane == 0) {
          if (j == 0 || mbar_wait(&bar.k_empty[c], (j - 1) & 1, abort))
            mbar_arrive_expect_tx(&bar.k_full[c], t.nloaded * seg_bytes);
        }
        __syncwarp();
        if (*abort) return;
        if (t.blk >= 0)
          tma_load_4d(sK + c * kChunkBytes + lane * G * 128, &p.kmap, &bar.k_full[c], c * 64, kvh, slot, t.blk);
      }
    };
    TileInfo cur = info(0);
    TileInfo nxt = info(1);
    load_k(0, cur);
    for (int j = 0; j < n_tiles && !*abort; ++j) {
      const int key0 = j * kBN;
      const int n_valid = min(kBN, seq_len - key0);
      if (cur.bad && lane == 0) record_error(p.dev_err, kErrDeviceBounds);
      // K of the next tile first: it streams in while QK_j runs (it waits only for QK_j)
      if (j + 1 < n_tiles) load_k(j + 1, nxt);
      __syncwarp();
      if (*abort) break;
      // V_j once PV_{j-1} has released the V tile
      if (lane == 0 && j > 0) mbar_wait(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort);
      __syncwarp();
      if (*abort) break;
      if (!cur.fix) {
        if (lane == 0) mbar_arrive_expect_tx(&bar.v_full, cur.big ? (uint32_t)kTileBytes : 4u * cur.nloaded * seg_bytes);
        __syncwarp();
        if (cur.big) issue_big(sV, &p.vmap_big, &bar.v_full, cur);
        else if (cur.blk >= 0) issue_seg(sV, &p.vmap, &bar.v_full, cur.blk, key0);
      } else {
        // V rows past seq_len or in a bad segment must be zero (P is 0 there, but 0 * NaN is not):
        // load through the private barrier, zero those rows, then publish.
        if (lane == 0) mbar_arrive_expect_tx(&bar.fix, cur.big ? (uint32_t)kTileBytes : 4u * cur.nloaded * seg_bytes);
        __syncwarp();
        if (cur.big) issue_big(sV, &p.vmap_big, &bar.fix, cur);
        else if (cur.blk >= 0) issue_seg(sV, &p.vmap, &bar.fix, cur.blk, key0);
        if (lane == 0) mbar_wait(&bar.fix, fix_phase & 1, abort);
        ++fix_phase;
        __syncwarp();
        if (*abort) break;
        zero_rows(sV, n_valid, cur.bad, G, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.v_full);
      }
      __syncwarp();
      cur = nxt;
      nxt = info(j + 2);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_f16(128, 128, !kInt8, false, false);
      constexpr uint32_t id_pv = idesc_f16(128, 256, true, false, true);
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
      bool ok = mbar_wait(kInt8 ? &bar.q_ready : &bar.q_full, 0, abort);
      auto issue_pv = [&](int i) -> bool {
        if (!mbar_wait(&bar.p_full[i & 1], (i >> 1) & 1, abort)) return false;
        if (!mbar_wait(&bar.v_full, i & 1, abort)) return false;
        tc_fence_after();
        const uint32_t a = tmem + ((i & 1) ? kColP1 : kColP0);
        for (int ks = 0; ks < 8; ++ks)
          umma_f16_ts(tmem + kColO, a + ks * 8, smem_desc(v_base + ks * 2048, 16384, 1024), id_pv,
                      (i > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&bar.pv_done[i & 1]);
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        // S is single-buffered: QK_j overwrites it once both softmax halves hold S_{j-1} in
        // registers (PV_{j-2}, queued before QK_j, keeps the tensor pipe busy meanwhile)
        if (j >= 1 && !mbar_wait(&bar.s_free, (j - 1) & 1, abort)) break;
        const uint32_t dS = tmem + kColS;
        for (int c = 0; c < 4; ++c) {
          if (!mbar_wait(&bar.k_full[c], j & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t off = c * kChunkBytes + kk * 32;
            umma_f16_ss(dS, smem_desc(q_base + off, 16, 1024), smem_desc(k_base + off, 16, 1024), id_qk,
                        (c | kk) ? 1u : 0u);
          }
          umma_commit(&bar.k_empty[c]);
        }
        if (!ok) break;
        umma_commit(&bar.s_full);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok && n_tiles > 0) issue_pv(n_tiles - 1);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------------------------- softmax
    // Two warpgroups share every row: half h = 0 owns score columns 0-63 and O columns 0-127,
    // half h = 1 columns 64-127 and O columns 128-255. Thread (h, i) owns row i = TMEM lane i.
    // Both halves meet at named barrier 1 (256 threads) a fixed number of times per tile; a
    // failed wait never skips a barrier - it only marks the warp dead, so the barriers stay paired.
    const int h = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;
    const int p_i = min(p0 + i, seq_len - 1);
    const bool row_valid = i < rows_valid;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float sc = p.scale_log2;
    bool dead = false;  // warp-uniform
    if (kInt8) {
      dead = !__all_sync(0xffffffffu, mbar_wait(&bar.q_full, 0, abort));
      if (!dead && h == 0) {
        bar.qscale[i] = quantize_q_row_inplace(sQ, i);
        fence_proxy_async_smem();
        mbar_arrive(&bar.q_ready);
      }
      if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(&bar.q_ready, 0, abort));
      if (!dead) sc = p.scale_log2 * bar.qscale[i];
    }
    float m_run = -INFINITY, l_run = 0.0f;
    for (int j = 0; j < n_tiles; ++j) {
      const int key0 = j * kBN;
      const float* ks = bar.kscale[j & 1] + 64 * h;
      if (kInt8 && h == 0 && !dead) {
        const int key = key0 + i;
        float v = 0.0f;
        if (key < seq_len) v = __ldg(p.k8_scale + ((int64_t)r * p.max_ctx + key) * p.num_kv_heads + kvh);
        bar.kscale[j & 1][i] = v;
      }
      if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(&bar.s_full, j & 1, abort));
      const uint32_t sb = tmem + lane_off + kColS;
      const uint32_t pb = tmem + lane_off + ((j & 1) ? kColP1 : kColP0);
      uint32_t sv[64];
      if (!dead) {
        tc_fence_after();
        uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        tmem_ld_32x32b_x32(sb + 64 * h, a);
        tmem_ld_32x32b_x32(sb + 64 * h + 32, b);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar.s_free);  // S may now be overwritten by QK_{j+1}
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = 0u;
      }
      const int lim = p_i - key0 - 64 * h;  // this half's columns > lim are masked
      const bool need_mask = lim < 63;
      if (kInt8) {  // fold the per-key scales in place: s = S * ks
        named_bar_sync(1, 256);  // this tile's kscale, written by half 0, is visible
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * ks[e]);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        float v = __uint_as_float(sv[e]);
        if (need_mask && e > lim) v = -INFINITY;
        mx = fmaxf(mx, v);
      }
      mx *= sc;  // sc > 0 (or NaN for a NaN q row)
      // both halves of a row agree on its maximum through shared memory
      bar.rowmax[j & 1][h][i] = mx;
      named_bar_sync(1, 256);
      mx = fmaxf(mx, bar.rowmax[j & 1][h ^ 1][i]);
      bool rescale = false;
      float alpha = 1.0f;
      if (m_run == -INFINITY || mx > m_run + kRescaleThreshold) {
        const float m_new = fmaxf(m_run, mx);
        if (m_new != -INFINITY) {
          rescale = m_run != -INFINITY;
          alpha = rescale ? ex2_approx(m_run - m_new) : 0.0f;
          l_run *= alpha;
          m_run = m_new;
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
      // P = exp2(s*sc - m) packed to bf16 pairs; the row sum uses the rounded weights that the PV
      // MMA multiplies, so the result is a convex combination of V rows
      uint32_t pk[32];
      float lsum = 0.0f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float s0 = __uint_as_float(sv[2 * e]), s1 = __uint_as_float(sv[2 * e + 1]);
        if (need_mask && 2 * e > lim) s0 = -INFINITY;
        if (need_mask && 2 * e + 1 > lim) s1 = -INFINITY;
        const float e0 = ex2_approx(fmaf(s0, sc, -m_use)), e1 = ex2_approx(fmaf(s1, sc, -m_use));
        pk[e] = pack_bf16x2(e0, e1);
        lsum += __uint_as_float(pk[e] << 16) + __uint_as_float(pk[e] & 0xffff0000u);
      }
      l_run += lsum;
      // P buffer j%2 was last read by PV_{j-2}; O may be rescaled only once PV_{j-1} is done
      if (!dead && j >= 2)
        dead = !__all_sync(0xffffffffu, mbar_wait(&bar.pv_done[j & 1], ((j - 2) >> 1) & 1, abort));
      const bool need_o = __any_sync(0xffffffffu, rescale);
      if (!dead && need_o && j >= 1)
        dead = !__all_sync(0xffffffffu, mbar_wait(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort));
      if (!dead) {
        tc_fence_after();
        tmem_st_32x32b_x32(pb + 32 * h, pk);  // P columns 32h..32h+31 = keys 64h..64h+63
        if (need_o) {
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            const uint32_t oa = tmem + lane_off + kColO + 128 * h + cc * 32;
            tmem_ld_32x32b_x32(oa, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st_32x32b_x32(oa, v);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar.p_full[j & 1]);
      }
    }
    // epilogue: O / l -> bf16, each half writes its 128 output columns of the row
    bool fin = !dead && !*abort && n_tiles > 0;
    if (n_tiles >= 2) fin = fin && mbar_wait(&bar.pv_done[n_tiles & 1], ((n_tiles - 2) >> 1) & 1, abort);
    fin = fin && mbar_wait(&bar.pv_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, abort);
    fin = __all_sync(0xffffffffu, fin);
    bar.rowmax[n_tiles & 1][h][i] = l_run;  // the slots of the parity no later tile reads
    named_bar_sync(1, 256);
    const float l_tot = l_run + bar.rowmax[n_tiles & 1][h ^ 1][i];
    if (fin) {
      tc_fence_after();
      const float inv_l = l_tot > 0.0f ? 1.0f / l_tot : 0.0f;
      uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(tok0 + i) * p.num_q_heads + qh) * kD + 128 * h);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_off + kColO + 128 * h + cc * 32, v);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * inv_l, __uint_as_float(v[8 * q + 1]) * inv_l);
            o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv_l, __uint_as_float(v[8 * q + 3]) * inv_l);
            o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv_l, __uint_as_float(v[8 * q + 5]) * inv_l);
            o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv_l, __uint_as_float(v[8 * q + 7]) * inv_l);
            dst[cc * 4 + q] = o;
          }
        }
      }
    }
  } else if (kFused && warp >= 12) {
    // ---------------------------------------------------------------------------- fp8 dequant
    // thread t owns key row t of each tile: its e4m3 K row (256 B) and V row are read straight from
    // the paged pool through the block table (64-bit offsets), dequantized exactly as
    // kv_fp8_dequant_dense does (bf16_rn(fp32(e4m3) * scale)) and written into the swizzled bf16
    // tiles: K chunk by chunk as QK_{j-1} releases it, V once PV_{j-1} is done. Rows past seq_len
    // or in an out-of-range block are zeros. The next row's loads are issued before each wait.
    const int t = (warp - 12) * 32 + lane;
    const float ksc = __ldg(p.k_scale), vsc = __ldg(p.v_scale);
    auto row_src = [&](const uint8_t* pool, int key) -> const uint4* {
      if (key >= seq_len) return nullptr;
      const int col = key / p.block_size;
      const int blk = col < p.max_blocks ? __ldg(p.block_table + (int64_t)r * p.bt_stride + col) : -1;
      if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        record_error(p.dev_err, kErrDeviceBounds);
        return nullptr;
      }
      return reinterpret_cast<const uint4*>(pool + (int64_t)blk * p.stride_blk +
                                            (int64_t)(key % p.block_size) * p.stride_tok +
                                            (int64_t)kvh * p.stride_head);
    };
    uint4 raw[16];
    auto load_row = [&](const uint4* src) {
#pragma unroll
      for (int q = 0; q < 16; ++q) raw[q] = src ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
    };
    // 64 codes of chunk c -> row t of chunk c of a swizzled [4][128][64 x bf16] tile
    auto store_chunk = [&](uint8_t* tile, int c, float sc) {
      uint8_t* row = tile + c * kChunkBytes + t * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 hi;
        const uint4 lo = dequant16_e4m3_bf16(raw[4 * c + q], sc, hi);
        *reinterpret_cast<uint4*>(row + (((2u * q) ^ (t & 7)) * 16)) = lo;
        *reinterpret_cast<uint4*>(row + (((2u * q + 1) ^ (t & 7)) * 16)) = hi;
      }
    };
    load_row(row_src(p.k_fp8, t));
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // unrolled: raw[] stays in registers
        if (j > 0 && !mbar_wait(&bar.k_empty[c], (j - 1) & 1, abort)) {
          ok = false;
          break;
        }
        store_chunk(sK, c, ksc);
        fence_proxy_async_smem();
        mbar_arrive(&bar.k_full[c]);
      }
      if (!ok) break;
      load_row(row_src(p.v_fp8, j * kBN + t));
      if (j > 0 && !mbar_wait(&bar.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort)) break;
#pragma unroll
      for (int c = 0; c < 4; ++c) store_chunk(sV, c, vsc);
      fence_proxy_async_smem();
      mbar_arrive(&bar.v_full);
      if (j + 1 < n_tiles) load_row(row_src(p.k_fp8, (j + 1) * kBN + t));
    }
  } else if (kConv && warp >= 12) {
    // ---------------------------------------------------------------------------- int8 K widening
    // thread t owns key row t of each tile: its 256 int8 codes come straight from the dense scratch
    // (16 x 16-byte loads, issued before waiting for the K tile to be free), are widened to fp16
    // integers and stored into the swizzled K tile chunk by chunk as QK_{j-1} releases it
    const int t = (warp - 12) * 32 + lane;
    for (int j = 0; j < n_tiles; ++j) {
      const int key = j * kBN + t;
      uint4 raw[16];
      if (key < seq_len) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.k8 + (((int64_t)r * p.max_ctx + key) * p.num_kv_heads + kvh) * kD);
#pragma unroll
        for (int q = 0; q < 16; ++q) raw[q] = __ldg(src + q);
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) raw[q] = make_uint4(0, 0, 0, 0);
      }
      bool ok = true;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (j > 0 && !mbar_wait(&bar.k_empty[c], (j - 1) & 1, abort)) {
          ok = false;
          break;
        }
        uint8_t* row = sK + c * kChunkBytes + t * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 16 codes = fp16 elements 64c + 16q .. +15
          uint4 lo, hi;
          widen16(raw[4 * c + q], lo, hi);
          *reinterpret_cast<uint4*>(row + (((2u * q) ^ (t & 7)) * 16)) = lo;
          *reinterpret_cast<uint4*>(row + (((2u * q + 1) ^ (t & 7)) * 16)) = hi;
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar.k_full[c]);
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && bar.abort) record_error(p.dev_err, kErrTimeout);
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

extern "C" pkv_status pkv_paged_prefill_attn(const void* q, const void* k_cache, const void* v_cache,
                                             int64_t num_blocks, int64_t stride_blk, int64_t stride_tok,
                                             int64_t stride_head, const int32_t* block_table, int64_t bt_stride,
                                             int32_t max_blocks, const int32_t* seq_lens,
                                             const int32_t* query_start_loc, int32_t num_reqs, int32_t total_q,
                                             int32_t max_q_len, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t block_size, float softmax_scale,
                                             int32_t qk_mode, const int8_t* k8, const float* k8_scale,
                                             const void* k16, int64_t max_ctx, void* out, int32_t* dev_err,
                                             void* stream) {
  using namespace pkv;
  clear_error();
  PKV_UNSUP(head_dim == kD, "paged_prefill_attn: head_dim must be 256 (got %d)", head_dim);
  PKV_ARG(qk_mode == PKV_QK_BF16 || qk_mode == PKV_QK_INT8, "paged_prefill_attn: unknown qk_mode %d", qk_mode);
  const bool int8 = qk_mode == PKV_QK_INT8;
  if (num_reqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;  // nothing to do, nothing read
  PKV_ARG(q && v_cache && block_table && seq_lens && query_start_loc && out,
          "paged_prefill_attn: null pointer argument");
  PKV_ARG(int8 ? ((k8 || k16) && k8_scale && max_ctx > 0) : (k_cache != nullptr),
          "paged_prefill_attn: missing K source for the selected qk_mode");
  PKV_ARG(num_reqs >= 0 && total_q >= 0 && max_q_len >= 0 && num_blocks > 0 && block_size > 0 &&
              max_blocks > 0 && bt_stride >= max_blocks && num_q_heads > 0 && num_kv_heads > 0,
          "paged_prefill_attn: bad size argument");
  PKV_UNSUP(num_q_heads % num_kv_heads == 0, "paged_prefill_attn: num_q_heads %% num_kv_heads != 0");
  PKV_UNSUP(block_size % 8 == 0, "paged_prefill_attn: block_size must be a multiple of 8 (got %d)", block_size);
  PKV_ARG(stride_blk > 0 && stride_tok > 0 && stride_head > 0, "paged_prefill_attn: strides must be positive");
  PKV_ARG(aligned16(q) && aligned16(v_cache) && aligned16(out) && (int8 || aligned16(k_cache)) &&
              (!int8 || k16 || aligned16(k8)) && (!int8 || !k16 || aligned16(k16)) && stride_blk % 8 == 0 && stride_tok % 8 == 0 && stride_head % 8 == 0,
          "paged_prefill_attn: q, caches, out and strides must be 16-byte aligned");
  PKV_ARG(softmax_scale > 0.0f, "paged_prefill_attn: softmax_scale must be positive");
  PKV_UNSUP(!int8 || (int64_t)num_reqs * max_ctx < (1ll << 31), "paged_prefill_attn: int8 scratch too large");
  if (num_reqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;

  Params p{};
  const int G = gcd_int(block_size, kBN);
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)num_q_heads, (uint64_t)total_q};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)num_q_heads * kD * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kBM};
    pkv_status s = encode_tiled(&p.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, "q");
    if (s != PKV_OK) return s;
  }
  {
    const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)num_kv_heads, (uint64_t)block_size, (uint64_t)num_blocks};
    const uint64_t strides[3] = {(uint64_t)stride_head * 2, (uint64_t)stride_tok * 2, (uint64_t)stride_blk * 2};
    const uint32_t box[4] = {64, 1, (uint32_t)G, 1};
    pkv_status s = encode_tiled(&p.vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v_cache, dims, strides, box, "v_cache");
    if (s != PKV_OK) return s;
    if (!int8) {
      s = encode_tiled(&p.kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k_cache, dims, strides, box, "k_cache");
      if (s != PKV_OK) return s;
    }
    p.big_ok = block_size >= kBN;
    if (p.big_ok) {
      const uint32_t big[4] = {64, 1, (uint32_t)kBN, 1};
      s = encode_tiled(&p.vmap_big, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v_cache, dims, strides, big, "v_cache");
      if (s != PKV_OK) return s;
      if (!int8) {
        s = encode_tiled(&p.kmap_big, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k_cache, dims, strides, big, "k_cache");
        if (s != PKV_OK) return s;
      }
    }
  }
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.num_q_heads = num_q_heads;
  p.group = num_q_heads / num_kv_heads;
  p.block_size = block_size;
  p.seg = G;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.k8_scale = k8_scale;
  p.k8 = k8;
  p.max_ctx = max_ctx;
  p.num_kv_heads = num_kv_heads;
  p.n_mtiles = (max_q_len + kBM - 1) / kBM;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.dev_err = dev_err;

  dim3 grid((unsigned)p.n_mtiles, (unsigned)num_q_heads, (unsigned)num_reqs);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int mode = !int8 ? 0 : (k16 ? 2 : 1);
  if (mode == 2) {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)num_kv_heads, (uint64_t)num_reqs * (uint64_t)max_ctx};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)num_kv_heads * kD * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kBN};
    pkv_status s = encode_tiled(&p.k16map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, k16, dims, strides, box, "k16");
    if (s != PKV_OK) return s;
  }
  auto launch = [&](auto kernel, int threads, int smem_bytes, bool& attr) {
    if (!attr) {
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
      attr = true;
    }
    kernel<<<grid, threads, smem_bytes, st>>>(p);
  };
  static bool attr0 = false, attr1 = false, attr2 = false;
  if (mode == 0) launch(paged_prefill_attn_kernel<0>, Cfg<0>::kThreads, Cfg<0>::kSmem, attr0);
  else if (mode == 1) launch(paged_prefill_attn_kernel<1>, Cfg<1>::kThreads, Cfg<1>::kSmem, attr1);
  else launch(paged_prefill_attn_kernel<2>, Cfg<2>::kThreads, Cfg<2>::kSmem, attr2);
  return check_launch("paged_prefill_attn");
}

extern "C" pkv_status pkv_paged_prefill_attn_fp8(const void* q, const uint8_t* k_fp8, const uint8_t* v_fp8,
                                                 const float* k_scale, const float* v_scale, int64_t num_blocks,
                                                 int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                                 const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                                 const int32_t* seq_lens, const int32_t* query_start_loc,
                                                 int32_t num_reqs, int32_t total_q, int32_t max_q_len,
                                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t block_size, float softmax_scale, void* out,
                                                 int32_t* dev_err, void* stream) {
  using namespace pkv;
  clear_error();
  PKV_UNSUP(head_dim == kD, "paged_prefill_attn_fp8: head_dim must be 256 (got %d)", head_dim);
  if (num_reqs == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;  // nothing to do, nothing read
  PKV_ARG(q && k_fp8 && v_fp8 && k_scale && v_scale && block_table && seq_lens && query_start_loc && out,
          "paged_prefill_attn_fp8: null pointer argument");
  PKV_ARG(num_reqs > 0 && total_q > 0 && max_q_len > 0 && num_blocks > 0 && block_size > 0 && max_blocks > 0 &&
              bt_stride >= max_blocks && num_q_heads > 0 && num_kv_heads > 0,
          "paged_prefill_attn_fp8: bad size argument");
  PKV_UNSUP(num_q_heads % num_kv_heads == 0, "paged_prefill_attn_fp8: num_q_heads %% num_kv_heads != 0");
  PKV_ARG(stride_blk > 0 && stride_tok > 0 && stride_head > 0, "paged_prefill_attn_fp8: strides must be positive");
  PKV_ARG(aligned16(q) && aligned16(out) && aligned16(k_fp8) && aligned16(v_fp8) && stride_blk % 16 == 0 &&
              stride_tok % 16 == 0 && stride_head % 16 == 0,
          "paged_prefill_attn_fp8: q, out, pools and pool strides must be 16-byte aligned");
  PKV_ARG(softmax_scale > 0.0f, "paged_prefill_attn_fp8: softmax_scale must be positive");

  Params p{};
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)num_q_heads, (uint64_t)total_q};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)num_q_heads * kD * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kBM};
    pkv_status s = encode_tiled(&p.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, "q");
    if (s != PKV_OK) return s;
  }
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.num_q_heads = num_q_heads;
  p.group = num_q_heads / num_kv_heads;
  p.block_size = block_size;
  p.seg = gcd_int(block_size, kBN);
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.num_kv_heads = num_kv_heads;
  p.n_mtiles = (max_q_len + kBM - 1) / kBM;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.dev_err = dev_err;
  p.k_fp8 = k_fp8;
  p.v_fp8 = v_fp8;
  p.stride_blk = stride_blk;
  p.stride_tok = stride_tok;
  p.stride_head = stride_head;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(paged_prefill_attn_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<3>::kSmem);
    attr = true;
  }
  dim3 grid((unsigned)p.n_mtiles, (unsigned)num_q_heads, (unsigned)num_reqs);
  paged_prefill_attn_kernel<3><<<grid, Cfg<3>::kThreads, Cfg<3>::kSmem, static_cast<cudaStream_t>(stream)>>>(p);
  return check_launch("paged_prefill_attn_fp8");
}
