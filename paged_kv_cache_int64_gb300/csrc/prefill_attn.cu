// prefill_attn.cu - pkv_paged_prefill_attn: chunked causal prefill attention over a paged bf16
// KV cache, exact-QK (bf16) or int8-QK.
//
// HyperQwen PR #109 (_prefill_attn_kernel in prefill_attn_hd256.py; review: the "int8_qk=False"
// and "int8_qk=True" arms, chunk 2048, head_dim 256, block 880): for every query of the chunk,
// softmax(scale * q.K^T) V over the keys at or before its position, K and V read through the
// block table with the block id widened to int64 before the stride product.
//
// sm_103a design (one CTA = 128 query rows of one query head of one request):
//   warp 0      TMA producer: Q once; per key tile, K and V gathered from the paged pool with
//               4-D tensor maps [head_dim, kv_heads, block_size, num_blocks] whose block
//               coordinate is the block id (the TMA unit forms the 64-bit address): a tile inside
//               one block is 4 copies of 128 rows per tensor; with blocks under 128 keys a tile is
//               split into segments of gcd(block_size, 128) keys, one lane per segment reading the
//               table; the next tile's block ids are read early. Key tiles are 128 keys, or (kA:
//               block_size >= 128 and not a multiple of 128) follow the blocks, the last tile of a
//               block short, so that no tile straddles two blocks (tile_range, TileCursor).
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
//               rows in place first and loads each tile's per-key K scales a tile ahead. Q8.K8 runs as an f16 MMA: every product and partial sum is an
//               integer below 2^24, so the f32 accumulator holds the exact integer dot product.
// Rows of the last tile past seq_len (and of any out-of-range block) are zero-filled in shared
// memory before the MMAs read them, so stale or NaN pool bytes never reach P.V. Every wait is
// bounded: on expiry the CTA records PKV_ERR_TIMEOUT, drains and exits.
//
// Launches. Classic (no workspace): one CTA per (m-tile, head, request); the CTAs of one chunk all
// but tie in work, so 256 of them on 152 SMs leave the second wave 68% full. Persistent (a
// workspace given): one CTA per SM walks a static schedule of segments - whole units (request,
// m-tile, head) in full waves, then the units of the last partial wave cut into k equal key ranges
// so that their pieces fill every SM (SegIter). Both keep the CTAs sweeping the same keys at the
// same time, which is what lets 152 CTAs share every K/V tile through L2 (a stream-K split into
// equal contiguous shares starts each CTA at a different key offset, and measured slower for that
// reason). A piece writes the fp32 O / l of its keys and the rows' log-sum-exp to the workspace;
// prefill_combine_kernel merges the pieces into the bf16 rows. Every role walks the same
// segments; barrier phases follow the CTA's running tile count, positions and masks the tile index
// within the unit. Between segments, Q is reloaded once the last QK has read it (q_empty) and the
// first PV of the next unit overwrites O once the epilogue has read it (o_free).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

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
// Units whose first query row sees at most kLoKeys keys take P as two bf16 parts, P = hi + lo with
// lo = bf16(P - hi), and O += hi V + lo V (16 PV MMAs instead of 8). A bf16 weight alone carries a
// relative error up to 2^-9; over many keys these errors average out in the output, over a few they
// do not (rows with a handful of visible keys would miss the output bar by up to 2x). With the
// remainder the weights are exact to ~2^-17. Only the first query tiles of a prompt's first chunk
// qualify, so the cost stays there.
constexpr int kLoKeys = 1024;

// dynamic shared memory layout (1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kTilesEnd = kOffV + kTileBytes;

struct Barriers {
  uint64_t q_full;      // TMA Q landed (phase = segment parity)
  uint64_t q_ready;     // int8: Q quantized in place
  uint64_t q_empty;     // the segment's last QK has read Q: the next segment's Q may land
  uint64_t o_free;      // the segment's epilogue has read O (256 softmax arrivals)
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
  uint64_t drain;       // after a wait gave up: every MMA issued so far is complete
  uint32_t armed[7];    // phases the producer started (TMA or its own arrival): q_full, k_full[0..3],
                        // v_full, fix - the drain waits for the last one of each
  uint32_t tmem_base;
  int abort;
  float kscale[2][kBN];  // int8: per-key scales of the tile
  float qscale[kBM];     // int8: per-row q scales
  float rowmax[2][2][kBM];  // per tile parity, per half: row maxima
  float lsum[2][kBM];       // per half: the segment's row sums (epilogue)
};

// workspace of the persistent launch: kMaxSplit slots per CTA (the pieces of the units cut in key
// ranges, fewer than P units of at most kMaxSplit pieces), each the normalised fp32 O [128 rows][256]
// followed by the rows' natural-log LSE [128]. The last slot (never a piece's: pieces number at most
// (P - 1) kMaxSplit) holds the merge's header: F, R, k, then per cut unit its tok0, head, rows and
// key tiles, written by the persistent kernel so that the merge need not recompute the schedule.
constexpr int kMaxSplit = 4;
constexpr int64_t kSlotFloats = (int64_t)kBM * kD + kBM;
constexpr int64_t kCtaWsBytes = kMaxSplit * kSlotFloats * 4;
constexpr int kHdrUnits = 4;  // ints before the first unit entry

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
  // persistent launch: num_ctas CTAs walk the schedule of whole units and key-range pieces
  int32_t persistent;
  int32_t num_reqs;
  int32_t num_ctas;  // the persistent grid
  int32_t total_q;
  // key tiles: 0 - tile t holds keys [128 t, 128 t + 128); else (block_size >= 128 and not a multiple
  // of 128) the tiles of each block in turn, tpb = ceil(block_size / 128) per block, the last one
  // short, so that no tile straddles two blocks
  int32_t tpb;
  float tpb_inv;  // 1 / tpb (fast division of tile indices)
  float* ws;         // [num_ctas * kMaxSplit][kSlotFloats]
  uint64_t wait_limit_ns;  // bound on each wait (kWaitLimitNs unless a test shortens it)
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

// The same exp2 instruction as ex2_approx (so the same result bit for bit), marked volatile so that
// the compiler recomputes it instead of keeping 64 earlier results alive across a wait.
__device__ __forceinline__ float ex2_again(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// A unit of work: 128 query rows (m-tile mt) of query head qh of request r.
struct Unit {
  int r, qh, mt, kvh, seq_len, rows_valid, p0, n_tiles, tok0;
  bool lo;  // P as two bf16 parts (p0 < kLoKeys)
};

// Key tiles. With p.tpb == 0 tile t is keys [128 t, 128 t + 128). Otherwise tiles follow the blocks:
// tile t is the (t % tpb)-th 128-key piece of block t / tpb, the block's last piece shorter, so a
// tile never straddles two blocks and is always one TMA box per chunk (the box's rows past the
// block end read as zeros and are masked). With block_size 880 this removes the 16-key segment
// loads that one tile in eight would otherwise need.
// t = b * tpb + l (tile indices are below 2^24 since keys are below 2^31: the float quotient is
// within one of the exact one, and one correction step makes it exact)
__device__ __forceinline__ void tile_divmod(const Params& p, int t, int& b, int& l) {
  b = (int)((float)t * p.tpb_inv);
  l = t - b * p.tpb;
  if (l < 0) {
    --b;
    l += p.tpb;
  } else if (l >= p.tpb) {
    ++b;
    l -= p.tpb;
  }
}
// first key and number of keys of tile t
template <bool kA>
__device__ __forceinline__ void tile_range(const Params& p, int t, int& key0, int& len) {
  if constexpr (!kA) {
    key0 = t * kBN;
    len = kBN;
    return;
  }
  int b, l;
  tile_divmod(p, t, b, l);
  key0 = b * p.block_size + l * kBN;
  len = min(kBN, p.block_size - l * kBN);
}
// Walks consecutive tiles without divisions: the next tile starts where this one ends.
struct TileCursor {
  int key0, len;  // first key and number of keys of the tile
  int l;          // its index within its block (tpb > 0)
};
template <bool kA>
__device__ __forceinline__ TileCursor tile_cursor(const Params& p, int t) {
  TileCursor c;
  c.l = 0;
  if constexpr (kA) {
    int b;
    tile_divmod(p, t, b, c.l);
  }
  tile_range<kA>(p, t, c.key0, c.len);
  return c;
}
template <bool kA>
__device__ __forceinline__ void tile_advance(const Params& p, TileCursor& c) {
  c.key0 += c.len;
  if constexpr (kA) {
    if (++c.l == p.tpb) c.l = 0;
    c.len = min(kBN, p.block_size - c.l * kBN);
  }
}
// tiles covering keys [0, keys)
template <bool kA>
__device__ __forceinline__ int tiles_for(const Params& p, int keys) {
  if constexpr (!kA) return (keys + kBN - 1) / kBN;
  const int full = keys / p.block_size;
  return full * p.tpb + (keys - full * p.block_size + kBN - 1) / kBN;
}

// Fills u for (r, mt, qh); false when the m-tile holds no query rows.
template <bool kA>
__device__ __forceinline__ bool make_unit(const Params& p, int r, int mt, int qh, Unit& u) {
  const int q0 = __ldg(p.qsl + r);
  const int q_len = __ldg(p.qsl + r + 1) - q0;
  const int seq_len = __ldg(p.seq_lens + r);
  if (mt * kBM >= q_len || q_len > seq_len) return false;
  u.r = r;
  u.qh = qh;
  u.mt = mt;
  u.kvh = qh / p.group;
  u.seq_len = seq_len;
  u.rows_valid = min(kBM, q_len - mt * kBM);
  u.p0 = seq_len - q_len + mt * kBM;                      // position of row 0
  const int kv_end = min(seq_len, u.p0 + u.rows_valid);  // keys [0, kv_end)
  u.n_tiles = tiles_for<kA>(p, kv_end);
  u.tok0 = q0 + mt * kBM;
  u.lo = u.p0 < kLoKeys;
  return true;
}

// key tiles of each unit of (request r, m-tile mt); 0 when the m-tile holds no rows
template <bool kA>
__device__ __forceinline__ int unit_tiles(const Params& p, int r, int mt) {
  Unit u;
  return make_unit<kA>(p, r, mt, 0, u) ? u.n_tiles : 0;
}

// A segment: key tiles [t0, t1) of one unit, processed by this CTA.
struct Seg {
  Unit u;
  int t0, t1;
  bool whole;  // all of the unit's tiles: the CTA writes the final output rows
  int slot;    // otherwise the workspace slot of the piece
};

// The persistent schedule. Units with rows - groups (m-tile, request) in the order m-tile
// descending (heaviest first), then request, each group the num_q_heads units of its heads - are
// numbered u = 0 .. U - 1. With P CTAs, the first F = P floor(U / P) units are whole: CTA c takes
// units c, c + P, ... (full waves: every CTA sweeps its unit's keys from the first tile, in step
// with the others, so the K/V tiles they share are read from L2). The R = U - F remaining units
// (R < P) are each cut into k equal key ranges, k <= kMaxSplit chosen to fill the P CTAs: piece
// pi = i R + j is range i of unit F + j, and goes to CTA P - 1 - (pi mod P) (the CTAs holding the
// lightest whole units take the extra piece). Pieces in that order sweep the same key range at the
// same time, again in step; their fp32 partials land in workspace slot pi.
struct Schedule {
  int U, f, R, k;
};

template <bool kA>
__device__ int count_groups(const Params& p) {
  int n = 0;
  for (int m = p.n_mtiles - 1; m >= 0; --m)
    for (int r = 0; r < p.num_reqs; ++r) n += unit_tiles<kA>(p, r, m) > 0;
  return n;
}

// k in [1, kMaxSplit] minimising the time of the cut units' pieces, ceil(R k / P) / k waves of
// whole-unit time, plus 2% of a wave per extra piece (its epilogue, Q load and merge)
__host__ __device__ inline int choose_split(int R, int P) {
  int best = 1;
  float best_cost = 2.0f;
  for (int k = 1; k <= kMaxSplit && R > 0; ++k) {
    const float cost = (float)((R * k + P - 1) / P) / (float)k + 0.02f * (float)(k - 1);
    if (cost < best_cost - 1e-6f) {
      best_cost = cost;
      best = k;
    }
  }
  return best;
}

template <bool kA>
__device__ Schedule make_schedule(const Params& p) {
  Schedule sc;
  const int P = p.num_ctas;
  sc.U = count_groups<kA>(p) * p.num_q_heads;
  sc.f = sc.U / P;
  sc.R = sc.U - sc.f * P;
  sc.k = choose_split(sc.R, P);
  return sc;
}

// unit u of the persistent order
template <bool kA>
__device__ void unit_at(const Params& p, int u, Unit& out) {
  int g = u / p.num_q_heads;
  const int qh = u - g * p.num_q_heads;
  for (int m = p.n_mtiles - 1; m >= 0; --m)
    for (int r = 0; r < p.num_reqs; ++r)
      if (unit_tiles<kA>(p, r, m) > 0 && g-- == 0) {
        make_unit<kA>(p, r, m, qh, out);
        return;
      }
}

// Walks this CTA's segments; every role walks the same sequence. Classic launch: one segment, the
// unit of blockIdx (latest m-tiles first), whole. Persistent launch: its whole units, then its pieces.
template <bool kA>
struct SegIter {
  const Params& p;
  Schedule sc{};
  int count = 0;   // segments produced
  int w = 0;       // whole units taken
  int64_t pi = 0;  // next piece
  __device__ explicit SegIter(const Params& pp) : p(pp) {
    if (!p.persistent) return;
    sc = make_schedule<kA>(p);
    pi = p.num_ctas - 1 - (int)blockIdx.x;
  }
  __device__ bool next(Seg& s) {
    if (!p.persistent) {
      if (count++ > 0) return false;
      if (!make_unit<kA>(p, blockIdx.z, p.n_mtiles - 1 - (int)blockIdx.x, blockIdx.y, s.u)) return false;
      s.t0 = 0;
      s.t1 = s.u.n_tiles;
      s.whole = true;
      s.slot = 0;
      return s.u.n_tiles > 0;
    }
    const int P = p.num_ctas;
    if (w < sc.f) {
      unit_at<kA>(p, (int)blockIdx.x + P * w++, s.u);
      s.t0 = 0;
      s.t1 = s.u.n_tiles;
      s.whole = true;
      s.slot = 0;
      ++count;
      return true;
    }
    while (pi < (int64_t)sc.R * sc.k) {
      const int j = (int)(pi % sc.R), i = (int)(pi / sc.R);
      s.slot = (int)pi;
      pi += P;
      unit_at<kA>(p, sc.f * P + j, s.u);
      s.t0 = s.u.n_tiles * i / sc.k;
      s.t1 = s.u.n_tiles * (i + 1) / sc.k;
      if (s.t0 == s.t1) continue;  // a unit of fewer than k tiles: this range is empty
      s.whole = sc.k == 1;
      ++count;
      return true;
    }
    return false;
  }
};

// The roles of one CTA (producer, MMA issuer, softmax, converters). kLoCapable: some unit of this CTA
// takes P in two parts (its first row sees at most kLoKeys keys); the instantiation without it has
// none of that code, which would otherwise cost the common path about a fifth of its time.
template <int kMode, bool kA, bool kLoCapable>
__device__ __forceinline__ void cta_roles(const Params& p, uint8_t* smem, Barriers& bar, uint32_t tmem,
                                          volatile int* abort, uint64_t wl, int warp, int lane) {
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;
  constexpr bool kInt8 = kMode == 1 || kMode == 2;  // int8 QK (quantized Q, per-key K scales, f16 MMA)
  constexpr bool kConv = kMode == 1;                 // K widened by the converter warps
  constexpr bool kFused = kMode == 3;                // K and V dequantized by the converter warps
  if (warp == 0) {
    // ---------------------------------------------------------------------------- producer
    const int G = p.seg;
    const int nseg = kBN / G;
    const uint32_t seg_bytes = (uint32_t)G * 128u;  // one chunk of one segment
    if (lane == 0) {
      prefetch_tensormap(&p.qmap);
      if (!kFused) {
        prefetch_tensormap(&p.vmap);
        if (!kInt8) prefetch_tensormap(&p.kmap);
        if (kMode == 2) prefetch_tensormap(&p.k16map);
        if (p.big_ok) {
          prefetch_tensormap(&p.vmap_big);
          if (!kInt8) prefetch_tensormap(&p.kmap_big);
        }
      }
    }
    // Every go / stop decision of this warp is lane 0's wait result broadcast by one shuffle, so
    // the lanes never part (once any role gives up, every wait returns false promptly).
    auto uniform = [&](bool ok0) -> bool { return __shfl_sync(0xffffffffu, ok0, 0); };
    SegIter<kA> it(p);
    Seg sg;
    int g = 0, s = 0;
    uint32_t fix_phase = 0;
    bool go = true;
    while (go && it.next(sg)) {
      const Unit& u = sg.u;
      const int r = u.r, kvh = u.kvh, seq_len = u.seq_len;
      // Q of this segment's unit, once the previous segment's last QK has read the old one
      bool ok0 = true;
      if (lane == 0) {
        ok0 = s == 0 || mbar_wait(&bar.q_empty, (s - 1) & 1, abort, wl);
        if (ok0) {
          mbar_arm_tx(&bar.q_full, kTileBytes, &bar.armed[0]);
          for (int c = 0; c < 4; ++c) tma_load_3d(sQ + c * kChunkBytes, &p.qmap, &bar.q_full, c * 64, u.qh, u.tok0);
        }
      }
      if (!uniform(ok0)) break;
      if (kFused) {  // K and V come from the converter warps
        g += sg.t1 - sg.t0;
        ++s;
        continue;
      }
      // block id of segment `lane` of the tile with keys [key0, key0 + len): >= 0, -1 past the tile
      // or seq_len, -2 out-of-range entry
      auto lookup = [&](int key0, int len) -> int {
        const int pos = key0 + lane * G;
        if (lane >= nseg || lane * G >= len || pos >= seq_len) return -1;
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
        bool big;          // the tile's keys lie in one valid block: 4 copies of 128 rows per tensor
        int blk0, slot0;   // block and first slot of key 0 of the tile
        int key0, len;     // the tile's keys
      };
      // the tile at cursor c (in_seg: one of the segment's tiles)
      auto info = [&](const TileCursor& c, bool in_seg) -> TileInfo {
        TileInfo t;
        const int key0 = c.key0, len = c.len;
        t.key0 = key0;
        t.len = len;
        t.blk = in_seg ? lookup(key0, len) : -1;
        t.bad = __ballot_sync(0xffffffffu, t.blk == -2);
        t.nloaded = __popc(__ballot_sync(0xffffffffu, t.blk >= 0));
        t.fix = t.bad != 0 || seq_len - key0 < len;
        t.blk0 = __shfl_sync(0xffffffffu, t.blk, 0);
        t.slot0 = key0 % p.block_size;
        // one block holds the tile's keys: 4 copies of a 128-row box per tensor (rows past the
        // block's end, in a short tile, read as zeros)
        t.big = p.big_ok && t.bad == 0 && t.blk0 >= 0 && t.slot0 + len <= p.block_size;
        return t;
      };
      // a whole tile of one tensor with 4 copies of [128 rows][64 x 16-bit] (lane 0)
      auto issue_big = [&](uint8_t* tile, const CUtensorMap* map, uint64_t* mb, const TileInfo& t) {
        if (lane == 0)
          for (int c = 0; c < 4; ++c) tma_load_4d(tile + c * kChunkBytes, map, mb, c * 64, kvh, t.slot0, t.blk0);
      };
      // K of the tile t (CTA tile gk) chunk by chunk as QK_{gk-1} frees it. K rows past seq_len need no
      // zero-fill (their scores are masked); rows of a bad segment do, so such a tile goes through
      // the private barrier, is patched, then published.
      // returns false (the same in every lane) when a wait gave up
      auto load_k = [&](int gk, const TileInfo& t) -> bool {
        const int key0 = t.key0;
        if (kConv) return true;  // the converter warps read the int8 K rows themselves
        if (kMode == 2) {        // fp16 copy of the int8 codes, dense by position: 4 copies of 128 rows
          bool ok0 = true;
          if (lane == 0) {
            const int row = (int)((int64_t)r * p.max_ctx + key0);
            for (int c = 0; c < 4 && ok0; ++c) {
              ok0 = gk == 0 || mbar_wait(&bar.k_empty[c], (gk - 1) & 1, abort, wl);
              if (!ok0) break;
              mbar_arm_tx(&bar.k_full[c], (uint32_t)kChunkBytes, &bar.armed[1 + c]);
              tma_load_3d(sK + c * kChunkBytes, &p.k16map, &bar.k_full[c], c * 64, kvh, row);
            }
          }
          return uniform(ok0);
        }
        if (t.bad) {
          // the copies follow their arming whatever happens meanwhile (the drain waits for them)
          bool ok0 = true;
          if (lane == 0) {
            for (int c = 0; c < 4 && gk > 0 && ok0; ++c) ok0 = mbar_wait(&bar.k_empty[c], (gk - 1) & 1, abort, wl);
            if (ok0) mbar_arm_tx(&bar.fix, 4u * t.nloaded * seg_bytes, &bar.armed[6]);
          }
          if (!uniform(ok0)) return false;
          if (t.blk >= 0) issue_seg(sK, &p.kmap, &bar.fix, t.blk, key0);
          if (lane == 0) ok0 = mbar_wait(&bar.fix, fix_phase & 1, abort, wl);
          ++fix_phase;
          if (!uniform(ok0)) return false;
          zero_rows(sK, kBN, t.bad, G, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0)
            for (int c = 0; c < 4; ++c) {
              mbar_arrive(&bar.k_full[c]);
              ++bar.armed[1 + c];  // as for V: counted for the drain's parity
            }
          __syncwarp();
          return true;
        }
        if (t.big) {
          bool ok0 = true;
          if (lane == 0) {
            for (int c = 0; c < 4; ++c) {
              ok0 = gk == 0 || mbar_wait(&bar.k_empty[c], (gk - 1) & 1, abort, wl);
              if (!ok0) break;
              mbar_arm_tx(&bar.k_full[c], (uint32_t)kChunkBytes, &bar.armed[1 + c]);
              tma_load_4d(sK + c * kChunkBytes, &p.kmap_big, &bar.k_full[c], c * 64, kvh, t.slot0, t.blk0);
            }
          }
          return uniform(ok0);
        }
        const int slot = (key0 + lane * G) % p.block_size;
        for (int c = 0; c < 4; ++c) {
          bool ok0 = true;
          if (lane == 0) {
            ok0 = gk == 0 || mbar_wait(&bar.k_empty[c], (gk - 1) & 1, abort, wl);
            if (ok0) mbar_arm_tx(&bar.k_full[c], t.nloaded * seg_bytes, &bar.armed[1 + c]);
          }
          if (!uniform(ok0)) return false;  // the copies follow their arming
          if (t.blk >= 0)
            tma_load_4d(sK + c * kChunkBytes + lane * G * 128, &p.kmap, &bar.k_full[c], c * 64, kvh, slot, t.blk);
        }
        return true;
      };
      TileCursor nc = tile_cursor<kA>(p, sg.t0);  // the tile `nxt` describes
      TileInfo cur = info(nc, true);
      tile_advance<kA>(p, nc);
      TileInfo nxt = info(nc, sg.t0 + 1 < sg.t1);
      go = load_k(g, cur);
      for (int j = sg.t0; go && j < sg.t1; ++j, ++g) {
        const int key0 = cur.key0;
        const int n_valid = min(cur.len, seq_len - key0);
        if (cur.bad && lane == 0) record_error(p.dev_err, kErrDeviceBounds);
        // K of the next tile first: it streams in while QK_g runs (it waits only for QK_g)
        if (j + 1 < sg.t1 && !(go = load_k(g + 1, nxt))) break;
        // V of tile g once PV_{g-1} has released the V tile
        bool ok0 = true;
        if (lane == 0 && g > 0) ok0 = mbar_wait(&bar.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort, wl);
        if (!(go = uniform(ok0))) break;
        if (!cur.fix) {
          if (lane == 0) mbar_arm_tx(&bar.v_full, cur.big ? (uint32_t)kTileBytes : 4u * cur.nloaded * seg_bytes, &bar.armed[5]);
          __syncwarp();
          if (cur.big) issue_big(sV, &p.vmap_big, &bar.v_full, cur);
          else if (cur.blk >= 0) issue_seg(sV, &p.vmap, &bar.v_full, cur.blk, key0);
        } else {
          // V rows past seq_len or in a bad segment must be zero (P is 0 there, but 0 * NaN is not):
          // load through the private barrier, zero those rows, then publish.
          if (lane == 0) mbar_arm_tx(&bar.fix, cur.big ? (uint32_t)kTileBytes : 4u * cur.nloaded * seg_bytes, &bar.armed[6]);
          __syncwarp();
          if (cur.big) issue_big(sV, &p.vmap_big, &bar.fix, cur);
          else if (cur.blk >= 0) issue_seg(sV, &p.vmap, &bar.fix, cur.blk, key0);
          if (lane == 0) ok0 = mbar_wait(&bar.fix, fix_phase & 1, abort, wl);
          ++fix_phase;
          if (!(go = uniform(ok0))) break;
          zero_rows(sV, n_valid, cur.bad, G, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bar.v_full);
            ++bar.armed[5];  // a phase the producer completed itself: counted for the drain's parity
          }
        }
        __syncwarp();
        cur = nxt;
        tile_advance<kA>(p, nc);
        nxt = info(nc, j + 2 < sg.t1);
      }
      ++s;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_f16(128, 128, !kInt8, false, false);
      constexpr uint32_t id_pv = idesc_f16(128, 256, true, false, true);
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
      // PV of CTA tile i; `first`: the first tile of segment si (O starts from zero once the
      // previous segment's epilogue has read it); `lo`: P is in two parts, hi in the first P buffer
      // and the remainder in the second, both multiplied into O
      auto issue_pv = [&](int i, bool first, int si, bool lo) -> bool {
        if (!mbar_wait(&bar.p_full[i & 1], (i >> 1) & 1, abort, wl)) return false;
        if (!mbar_wait(&bar.v_full, i & 1, abort, wl)) return false;
        if (first && si > 0 && !mbar_wait(&bar.o_free, (si - 1) & 1, abort, wl)) return false;
        tc_fence_after();
        const uint32_t a = tmem + ((lo || !(i & 1)) ? kColP0 : kColP1);
        for (int ks = 0; ks < 8; ++ks)
          umma_f16_ts(tmem + kColO, a + ks * 8, smem_desc(v_base + ks * 2048, 16384, 1024), id_pv,
                      (!first || ks > 0) ? 1u : 0u);
        if (lo)
          for (int ks = 0; ks < 8; ++ks)
            umma_f16_ts(tmem + kColO, tmem + kColP1 + ks * 8, smem_desc(v_base + ks * 2048, 16384, 1024), id_pv, 1u);
        umma_commit(&bar.pv_done[i & 1]);
        return true;
      };
      SegIter<kA> it(p);
      Seg sg;
      int g = 0, s = 0;
      bool ok = true;
      int pend = -1;            // CTA tile of the PV not yet issued
      bool pend_first = false;  // ... the first tile of its segment
      int pend_seg = 0;         // ... in segment pend_seg
      bool pend_lo = false;     // ... of a unit with two-part P
      while (ok && it.next(sg)) {
        if (!mbar_wait(kInt8 ? &bar.q_ready : &bar.q_full, s & 1, abort, wl)) break;
        for (int j = sg.t0; ok && j < sg.t1; ++j, ++g) {
          // S is single-buffered: QK_g overwrites it once both softmax halves hold S_{g-1} in
          // registers (PV_{g-2}, queued before QK_g, keeps the tensor pipe busy meanwhile)
          if (g >= 1 && !mbar_wait(&bar.s_free, (g - 1) & 1, abort, wl)) {
            ok = false;
            break;
          }
          const uint32_t dS = tmem + kColS;
          for (int c = 0; c < 4; ++c) {
            if (!mbar_wait(&bar.k_full[c], g & 1, abort, wl)) {
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
          if (j + 1 == sg.t1) umma_commit(&bar.q_empty);  // the segment's last read of Q
          if (pend >= 0 && !issue_pv(pend, pend_first, pend_seg, pend_lo)) ok = false;
          pend = g;
          pend_first = j == sg.t0;
          pend_seg = s;
          pend_lo = kLoCapable && sg.u.lo;
        }
        // int8: the softmax quantizes the next segment's Q only after this segment's epilogue, which
        // waits for its last PV - so that PV cannot wait for the next segment's first QK
        if (kInt8 && ok && pend >= 0) {
          ok = issue_pv(pend, pend_first, pend_seg, pend_lo);
          pend = -1;
        }
        ++s;
      }
      if (ok && pend >= 0) issue_pv(pend, pend_first, pend_seg, pend_lo);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------------------------- softmax
    // Two warpgroups share every row: half h = 0 owns score columns 0-63 and O columns 0-127,
    // half h = 1 columns 64-127 and O columns 128-255. Thread (h, i) owns row i = TMEM lane i.
    // The two threads of a row (warps q and q + 4, TMEM lane quarter q) meet at named barrier 2 + q
    // (64 threads) once per tile and once per epilogue; int8 also has each half meet at barrier
    // 6 + h (128 threads) once per tile to share its keys' scales. A failed wait never skips a
    // barrier - it only marks the warp dead - so the barriers stay paired.
    const int h = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    bool dead = false;  // warp-uniform
    SegIter<kA> it(p);
    Seg sg;
    int g = 0, s = 0;
    while (it.next(sg)) {
      const Unit& u = sg.u;
      const int p_i = min(u.p0 + i, u.seq_len - 1);
      const bool row_valid = i < u.rows_valid;
      float sc = p.scale_log2;
      if (kInt8) {
        // half 0 quantizes the segment's Q rows in place; half 1 takes the row scales at the named
        // barrier (it never waits for q_full: with a one-tile segment the next segment's Q may land
        // before half 1 gets here, and a parity wait would then miss the phase)
        if (h == 0) {
          if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(&bar.q_full, s & 1, abort, wl));
          if (!dead) {
            bar.qscale[i] = quantize_q_row_inplace(sQ, i);
            fence_proxy_async_smem();
            mbar_arrive(&bar.q_ready);
          }
        }
        named_bar_sync(2 + quarter, 64);  // the two threads of row i: half 0 wrote its scale
        if (!dead) sc = p.scale_log2 * bar.qscale[i];
      }
      float m_run = -INFINITY, l_run = 0.0f;
      TileCursor tc = tile_cursor<kA>(p, sg.t0);
      // int8: thread i < 64 of half h loads the scale of key 64h + i of the tile at cursor c (0 past
      // a short tile or seq_len) - the keys of its own half's columns - one tile ahead, so the load's
      // latency stays off the path and only the half's own threads meet to share them
      const bool ks_loader = kInt8 && i < 64;
      auto key_scale = [&](const TileCursor& c) -> float {
        const int col = 64 * h + i;
        const int key = c.key0 + col;
        return (col < c.len && key < u.seq_len)
                   ? __ldg(p.k8_scale + ((int64_t)u.r * p.max_ctx + key) * p.num_kv_heads + u.kvh)
                   : 0.0f;
      };
      float ks_next = 0.0f;
      if (ks_loader && !dead) ks_next = key_scale(tc);
      for (int j = sg.t0; j < sg.t1; ++j, ++g, tile_advance<kA>(p, tc)) {
        const int key0 = tc.key0, len = tc.len;
        const float* ks = bar.kscale[g & 1] + 64 * h;
        if (ks_loader && !dead) {
          bar.kscale[g & 1][64 * h + i] = ks_next;
          if (j + 1 < sg.t1) {
            TileCursor nc = tc;
            tile_advance<kA>(p, nc);
            ks_next = key_scale(nc);
          }
        }
        if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(&bar.s_full, g & 1, abort, wl));
        // A two-part P takes both P buffers, which PV_{g-1} reads: such a unit waits for PV_{g-1}
        // (and so for every earlier PV) before it reads S, so that the two parts are stored as soon
        // as they are computed. The units before and after meet it only through its epilogue,
        // which waits for its last PV, so this wait never reaches across units.
        const bool lo = kLoCapable && u.lo;
        if (lo && !dead && g >= 1)
          dead = !__all_sync(0xffffffffu, mbar_wait(&bar.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort, wl));
        const uint32_t sb = tmem + lane_off + kColS;
        const uint32_t pb = tmem + lane_off + ((g & 1) ? kColP1 : kColP0);
        uint32_t sv[64];
        if (!dead) {
          tc_fence_after();
          uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
          uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
          tmem_ld_32x32b_x32(sb + 64 * h, a);
          tmem_ld_32x32b_x32(sb + 64 * h + 32, b);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bar.s_free);  // S may now be overwritten by QK_{g+1}
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) sv[e] = 0u;
        }
        // this half's columns > lim are masked: keys after the row's position or past a short tile
        const int lim = min(p_i, key0 + len - 1) - key0 - 64 * h;
        const bool need_mask = lim < 63;
        if (kInt8) {  // fold the per-key scales in place: s = S * ks
          named_bar_sync(6 + h, 128);  // this tile's scales of the half's keys, written by the half, are visible
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float a0, a1;
            mul2(a0, a1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), ks[e], ks[e + 1]);
            sv[e] = __float_as_uint(a0);
            sv[e + 1] = __float_as_uint(a1);
          }
        }
        // the masked scores become -inf in place, once, and only in warps that have some (tiles on
        // the diagonal or at a block's end); the loops below then need no mask
        if (__any_sync(0xffffffffu, need_mask)) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e > lim) sv[e] = 0xff800000u;  // -inf
        }
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e) mx = fmaxf(mx, __uint_as_float(sv[e]));
        mx *= sc;  // sc > 0 (or NaN for a NaN q row)
        // both halves of a row agree on its maximum through shared memory
        bar.rowmax[g & 1][h][i] = mx;
        named_bar_sync(2 + quarter, 64);  // the other thread of row i (same TMEM lane quarter)
        mx = fmaxf(mx, bar.rowmax[g & 1][h ^ 1][i]);
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
        // MMA multiplies, so the result is a convex combination of V rows. remainder: the second part
        // bf16(P - hi) of a two-part P, from hi in pk (the exp2 recomputed, bit for bit)
        // pairs e0 .. e0 + n - 1 (keys 2e, 2e + 1 of this half) into pk[0 .. n)
        auto pack_p = [&](uint32_t* pk, int e0, int n, bool remainder) -> float {
          float sa = 0.0f, sb = 0.0f;
#pragma unroll
          for (int k = 0; k < n; ++k) {
            const int e = e0 + k;
            float y0, y1;
            fma2(y0, y1, __uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]), sc, sc, -m_use, -m_use);
            if (remainder) {
              const float x0 = ex2_again(y0), x1 = ex2_again(y1);
              pk[k] = pack_bf16x2(x0 - __uint_as_float(pk[k] << 16), x1 - __uint_as_float(pk[k] & 0xffff0000u));
            } else {
              pk[k] = pack_bf16x2(ex2_approx(y0), ex2_approx(y1));
            }
            add_bf16x2_to(sa, sb, pk[k]);
          }
          return sa + sb;
        };
        uint32_t pk[32];
        float lsum = 0.0f;
        if (lo) {
          // every PV is done (waited above): both parts go to tensor memory as they are computed,
          // 16 words at a time so that the scores of the other half can die meanwhile
          if (!dead) {
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < 4; ++part) {
              uint32_t (&q)[8] = *reinterpret_cast<uint32_t(*)[8]>(&pk[8 * part]);
              lsum += pack_p(q, 8 * part, 8, false);
              tmem_st_32x32b_x8(tmem + lane_off + kColP0 + 32 * h + 8 * part, q);  // hi
              lsum += pack_p(q, 8 * part, 8, true);
              tmem_st_32x32b_x8(tmem + lane_off + kColP1 + 32 * h + 8 * part, q);  // remainder
            }
          }
        } else {
          lsum = pack_p(pk, 0, 32, false);
        }
        // P buffer g%2 was last read by PV_{g-2}; O may be rescaled only once PV_{g-1} is done
        // (never needed on a segment's first tile: the running max starts there)
        if (!dead && g >= 2 && !lo)
          dead = !__all_sync(0xffffffffu, mbar_wait(&bar.pv_done[g & 1], ((g - 2) >> 1) & 1, abort, wl));
        const bool need_o = __any_sync(0xffffffffu, rescale);
        if (!dead && need_o && g >= 1 && !lo)
          dead = !__all_sync(0xffffffffu, mbar_wait(&bar.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort, wl));
        if (!dead) {
          tc_fence_after();
          if (!lo) tmem_st_32x32b_x32(pb + 32 * h, pk);  // P columns 32h..32h+31 = keys 64h..64h+63
          if (need_o) {
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
              uint32_t v[32];
              const uint32_t oa = tmem + lane_off + kColO + 128 * h + cc * 32;
              tmem_ld_32x32b_x32(oa, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float a0, a1;
                mul2(a0, a1, __uint_as_float(v[e]), __uint_as_float(v[e + 1]), alpha, alpha);
                v[e] = __float_as_uint(a0);
                v[e + 1] = __float_as_uint(a1);
              }
              tmem_st_32x32b_x32(oa, v);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar.p_full[g & 1]);
        }
        l_run += lsum;
      }
      // epilogue: the segment's last PV done, then O / l - bf16 output rows for a whole unit, or
      // the normalised fp32 partial and its log-sum-exp for a unit cut between CTAs
      const int gl = g - 1;  // the segment's last CTA tile
      bool fin = !dead && !*abort && mbar_wait(&bar.pv_done[gl & 1], (gl >> 1) & 1, abort, wl);
      fin = __all_sync(0xffffffffu, fin);
      bar.lsum[h][i] = l_run;
      named_bar_sync(2 + quarter, 64);
      const float l_tot = l_run + bar.lsum[h ^ 1][i];
      if (fin) {
        tc_fence_after();
        const float inv_l = l_tot > 0.0f ? 1.0f / l_tot : 0.0f;
        if (sg.whole) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(u.tok0 + i) * p.num_q_heads + u.qh) * kD + 128 * h);
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
        } else {
          float* slot = p.ws + (int64_t)sg.slot * kSlotFloats;
          float4* dst = reinterpret_cast<float4*>(slot + (int64_t)i * kD + 128 * h);
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + lane_off + kColO + 128 * h + cc * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[cc * 8 + q] = make_float4(__uint_as_float(v[4 * q + 0]) * inv_l, __uint_as_float(v[4 * q + 1]) * inv_l,
                                            __uint_as_float(v[4 * q + 2]) * inv_l, __uint_as_float(v[4 * q + 3]) * inv_l);
          }
          // natural-log LSE of the row over this segment's keys: (m + log2 l) ln 2; -inf if none
          if (h == 0)
            slot[kBM * kD + i] = l_tot > 0.0f ? (m_run + __log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
          if (h == 0 && i == 0) {  // the unit's header entry (every piece writes the same values)
            int* e = reinterpret_cast<int*>(p.ws + ((int64_t)p.num_ctas * kMaxSplit - 1) * kSlotFloats) + kHdrUnits +
                     4 * (sg.slot % it.sc.R);
            e[0] = u.tok0;
            e[1] = u.qh;
            e[2] = u.rows_valid;
            e[3] = u.n_tiles;
          }
        }
      }
      if (!dead) {  // O has been read: the next segment's first PV may overwrite it
        tc_fence_before();
        mbar_arrive(&bar.o_free);
      }
      ++s;
    }
  } else if (kFused && warp >= 12) {
    // ---------------------------------------------------------------------------- fp8 dequant
    // thread t owns key row t of each tile: its e4m3 K row (256 B) and V row are read straight from
    // the paged pool through the block table (64-bit offsets), dequantized exactly as
    // kv_fp8_dequant_dense does (bf16_rn(fp32(e4m3) * scale)) and written into the swizzled bf16
    // tiles: K chunk by chunk as QK_{g-1} releases it, V once PV_{g-1} is done. Rows past seq_len
    // or in an out-of-range block are zeros. The next row's loads are issued before each wait.
    const int t = (warp - 12) * 32 + lane;
    const float ksc = __ldg(p.k_scale), vsc = __ldg(p.v_scale);
    uint4 raw[16];
    auto load_row = [&](const uint4* src) {
#pragma unroll
      for (int q = 0; q < 16; ++q) raw[q] = src ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
    };
    // 64 codes of chunk c -> row t of chunk c of a swizzled [4][128][64 x bf16] tile
    auto store_chunk = [&](uint8_t* tile, int c, float scv) {
      uint8_t* row = tile + c * kChunkBytes + t * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 hi;
        const uint4 lo = dequant16_e4m3_bf16(raw[4 * c + q], scv, hi);
        *reinterpret_cast<uint4*>(row + (((2u * q) ^ (t & 7)) * 16)) = lo;
        *reinterpret_cast<uint4*>(row + (((2u * q + 1) ^ (t & 7)) * 16)) = hi;
      }
    };
    SegIter<kA> it(p);
    Seg sg;
    int g = 0;
    bool ok = true;
    while (ok && it.next(sg)) {
      const Unit& u = sg.u;
      // row t of the tile at cursor c (nullptr: zeros - past a short tile, past seq_len, or a bad
      // block)
      auto row_src = [&](const uint8_t* pool, const TileCursor& c) -> const uint4* {
        const int key = c.key0 + t;
        if (t >= c.len || key >= u.seq_len) return nullptr;
        const int col = key / p.block_size;
        const int blk = col < p.max_blocks ? __ldg(p.block_table + (int64_t)u.r * p.bt_stride + col) : -1;
        if (blk < 0 || (int64_t)blk >= p.num_blocks) {
          record_error(p.dev_err, kErrDeviceBounds);
          return nullptr;
        }
        return reinterpret_cast<const uint4*>(pool + (int64_t)blk * p.stride_blk +
                                              (int64_t)(key % p.block_size) * p.stride_tok +
                                              (int64_t)u.kvh * p.stride_head);
      };
      TileCursor tc = tile_cursor<kA>(p, sg.t0);
      load_row(row_src(p.k_fp8, tc));
      for (int j = sg.t0; j < sg.t1 && ok; ++j, ++g) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // unrolled: raw[] stays in registers
          if (g > 0 && !mbar_wait(&bar.k_empty[c], (g - 1) & 1, abort, wl)) {
            ok = false;
            break;
          }
          store_chunk(sK, c, ksc);
          fence_proxy_async_smem();
          mbar_arrive(&bar.k_full[c]);
        }
        if (!ok) break;
        load_row(row_src(p.v_fp8, tc));
        if (g > 0 && !mbar_wait(&bar.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort, wl)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) store_chunk(sV, c, vsc);
        fence_proxy_async_smem();
        mbar_arrive(&bar.v_full);
        tile_advance<kA>(p, tc);
        if (j + 1 < sg.t1) load_row(row_src(p.k_fp8, tc));
      }
    }
  } else if (kConv && warp >= 12) {
    // ---------------------------------------------------------------------------- int8 K widening
    // thread t owns key row t of each tile: its 256 int8 codes come straight from the dense scratch
    // (16 x 16-byte loads, issued before waiting for the K tile to be free), are widened to fp16
    // integers and stored into the swizzled K tile chunk by chunk as QK_{g-1} releases it
    const int t = (warp - 12) * 32 + lane;
    SegIter<kA> it(p);
    Seg sg;
    int g = 0;
    bool ok = true;
    while (ok && it.next(sg)) {
      const Unit& u = sg.u;
      TileCursor tc = tile_cursor<kA>(p, sg.t0);
      for (int j = sg.t0; j < sg.t1 && ok; ++j, ++g, tile_advance<kA>(p, tc)) {
        const int key = tc.key0 + t;
        uint4 raw[16];
        if (t < tc.len && key < u.seq_len) {
          const uint4* src = reinterpret_cast<const uint4*>(
              p.k8 + (((int64_t)u.r * p.max_ctx + key) * p.num_kv_heads + u.kvh) * kD);
#pragma unroll
          for (int q = 0; q < 16; ++q) raw[q] = __ldg(src + q);
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) raw[q] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (g > 0 && !mbar_wait(&bar.k_empty[c], (g - 1) & 1, abort, wl)) {
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
      }
    }
  }
}

// Whether some unit of the launch may take P in two parts: a request with queries whose chunk starts
// before position kLoKeys (the same answer in every thread; a few loads per request). Launches of a
// prompt's later chunks answer no and run the instantiation without that code.
__device__ bool launch_has_lo_units(const Params& p) {
  const int n = p.persistent ? p.num_reqs : 1;
  const int r0 = p.persistent ? 0 : (int)blockIdx.z;
  for (int r = r0; r < r0 + n; ++r) {
    const int q_len = __ldg(p.qsl + r + 1) - __ldg(p.qsl + r);
    if (q_len > 0 && __ldg(p.seq_lens + r) - q_len < kLoKeys) return true;
  }
  return false;
}

// kA: key tiles follow the blocks (block_size >= 128, not a multiple of 128, several blocks per
// request); otherwise plain 128-key tiles
template <int kMode, bool kA>
__global__ void __launch_bounds__(Cfg<kMode>::kThreads, 1)
    paged_prefill_attn_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers& bar = *reinterpret_cast<Barriers*>(smem + Cfg<kMode>::kTiles);
  constexpr bool kConv = kMode == 1;                 // K widened by the converter warps
  constexpr bool kFused = kMode == 3;                // K and V dequantized by the converter warps

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (!p.persistent) {  // classic launch: a CTA without rows leaves at once (CTA-uniform)
    Unit u;
    if (!make_unit<kA>(p, blockIdx.z, p.n_mtiles - 1 - (int)blockIdx.x, blockIdx.y, u)) return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_ready, 128);
    mbar_init(&bar.q_empty, 1);
    mbar_init(&bar.o_free, 256);
    for (int c = 0; c < 4; ++c) {
      mbar_init(&bar.k_full[c], (kConv || kFused) ? 128 : 1);
      mbar_init(&bar.k_empty[c], 1);
    }
    mbar_init(&bar.v_full, kFused ? 128 : 1);
    mbar_init(&bar.fix, 1);
    mbar_init(&bar.drain, 1);
    for (int b = 0; b < 7; ++b) bar.armed[b] = 0;
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
  const uint64_t wl = p.wait_limit_ns;
  if (p.persistent && blockIdx.x == 0 && threadIdx.x == 96) {  // warp 3: the merge header's schedule
    const Schedule sc = make_schedule<kA>(p);
    int* hdr = reinterpret_cast<int*>(p.ws + ((int64_t)p.num_ctas * kMaxSplit - 1) * kSlotFloats);
    hdr[0] = sc.f * p.num_ctas;
    hdr[1] = sc.R;
    hdr[2] = sc.k;
  }
  // Barrier phases follow g, the CTA's running tile count over all its segments, and s, its
  // segment count; positions and masks follow the unit-local tile index j.

  if (launch_has_lo_units(p))
    cta_roles<kMode, kA, true>(p, smem, bar, tmem, abort, wl, warp, lane);
  else
    cta_roles<kMode, kA, false>(p, smem, bar, tmem, abort, wl, warp, lane);

  tc_fence_before();
  // every role has left its loop; the flag's final value, the same for every thread (a thread that
  // set it reads it set, so the OR over the CTA sees it)
  const bool gave_up = __syncthreads_or(*abort != 0);
  if (gave_up) {
    // some wait gave up: before the tensor memory is freed and the CTA exits, wait for what this
    // CTA still has in flight - the TMA copies of every phase it armed and every MMA it issued
    if (warp == 0 && lane == 0) {
      drain_armed(&bar.q_full, bar.armed[0]);
      for (int c = 0; c < 4; ++c) drain_armed(&bar.k_full[c], bar.armed[1 + c]);
      drain_armed(&bar.v_full, bar.armed[5]);
      drain_armed(&bar.fix, bar.armed[6]);
    }
    if (warp == 1 && lane == 0) {
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


// Merges the pieces of the units that the persistent launch cut into key ranges: block (b, y) takes
// rows 8y .. 8y + 7 of cut unit F + b. Piece i holds O_i = its keys' softmax-weighted V rows / l_i
// and lse_i = m_i + ln l_i; the row is sum_i e^(lse_i - M) O_i / sum_i e^(lse_i - M) with
// M = max_i lse_i (a piece whose keys the row cannot see has lse_i = -inf and weight 0). Warp w
// takes row 8y + w, lane l columns 8l .. 8l + 7; every load of the row is issued before the first
// is used (one memory round trip per thread).
constexpr int kCombineRows = 8;

__global__ void __launch_bounds__(256) prefill_combine_kernel(const __grid_constant__ Params p) {
  __shared__ Unit s_u;
  __shared__ int s_n;                          // pieces; 0: nothing to merge in this block
  __shared__ const float* s_slot[kMaxSplit];  // each piece's workspace slot
  // launched as a programmatic dependent: wait for the persistent kernel's writes
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    s_n = 0;
    const int* hdr = reinterpret_cast<const int*>(p.ws + ((int64_t)p.num_ctas * kMaxSplit - 1) * kSlotFloats);
    const int R = hdr[1], k = hdr[2];
    const int b = blockIdx.x;
    if (k > 1 && k <= kMaxSplit && R < p.num_ctas && b < R) {
      const int* e = hdr + kHdrUnits + 4 * b;
      Unit u;
      u.tok0 = e[0];
      u.qh = e[1];
      u.rows_valid = e[2];
      u.n_tiles = e[3];
      // the entry was written by this launch unless it aborted; never write outside out
      if (u.tok0 >= 0 && u.rows_valid >= 1 && u.rows_valid <= kBM && u.tok0 <= p.total_q - u.rows_valid &&
          u.qh >= 0 && u.qh < p.num_q_heads && u.n_tiles >= 1) {
        int n = 0;
        for (int i = 0; i < k; ++i)
          if (u.n_tiles * i / k < u.n_tiles * (i + 1) / k) s_slot[n++] = p.ws + ((int64_t)i * R + b) * kSlotFloats;
        s_u = u;
        s_n = n;
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  const int row = blockIdx.y * kCombineRows + (threadIdx.x >> 5);
  if (n == 0 || row >= s_u.rows_valid) return;
  const int lane = threadIdx.x & 31;
  float lse[kMaxSplit];
  float4 o[kMaxSplit][2];
#pragma unroll
  for (int k = 0; k < kMaxSplit; ++k) {
    if (k < n) {
      const float* sl = s_slot[k];
      lse[k] = sl[kBM * kD + row];
      const float4* src = reinterpret_cast<const float4*>(sl + (int64_t)row * kD) + 2 * lane;
      o[k][0] = src[0];
      o[k][1] = src[1];
    } else {
      lse[k] = -INFINITY;
      o[k][0] = o[k][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMaxSplit; ++k) M = fmaxf(M, lse[k]);
  float den = 0.0f;
  float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < kMaxSplit; ++k) {
    const float w = lse[k] == -INFINITY ? 0.0f : expf(lse[k] - M);
    den += w;
    acc[0] = fmaf(w, o[k][0].x, acc[0]);
    acc[1] = fmaf(w, o[k][0].y, acc[1]);
    acc[2] = fmaf(w, o[k][0].z, acc[2]);
    acc[3] = fmaf(w, o[k][0].w, acc[3]);
    acc[4] = fmaf(w, o[k][1].x, acc[4]);
    acc[5] = fmaf(w, o[k][1].y, acc[5]);
    acc[6] = fmaf(w, o[k][1].z, acc[6]);
    acc[7] = fmaf(w, o[k][1].w, acc[7]);
  }
  const float inv = den > 0.0f ? 1.0f / den : 0.0f;
  uint4 r;
  r.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  r.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
  r.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
  r.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
  reinterpret_cast<uint4*>(p.out + ((int64_t)(s_u.tok0 + row) * p.num_q_heads + s_u.qh) * kD)[lane] = r;
}

constexpr int kMaxCtas = 1024;  // persistent CTAs at most

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Launches mode kMode: the classic grid, or (workspace given) the persistent grid of
// P = min(SMs, workspace_bytes / kCtaWsBytes, kMaxCtas) CTAs followed by the combine ((P - 1) x 16
// blocks: at most P - 1 units are cut, 8 rows a block).
template <int kMode, bool kA>
pkv_status launch_prefill(Params& p, int32_t num_reqs, void* workspace, int64_t workspace_bytes, cudaStream_t st,
                          const char* name) {
  static std::atomic<uint64_t> attr_done{0};
  once_per_device(attr_done, [] {
    cudaFuncSetAttribute(paged_prefill_attn_kernel<kMode, kA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Cfg<kMode>::kSmem);
  });
  p.num_reqs = num_reqs;
  p.wait_limit_ns = take_wait_limit_ns();
  if (!workspace) {
    p.persistent = 0;
    dim3 grid((unsigned)p.n_mtiles, (unsigned)p.num_q_heads, (unsigned)num_reqs);
    paged_prefill_attn_kernel<kMode, kA><<<grid, Cfg<kMode>::kThreads, Cfg<kMode>::kSmem, st>>>(p);
    return check_launch(name);
  }
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t P = std::min<int64_t>({(int64_t)sms, workspace_bytes / kCtaWsBytes, (int64_t)kMaxCtas});
  p.persistent = 1;
  p.num_ctas = (int32_t)P;
  p.ws = static_cast<float*>(workspace);
  paged_prefill_attn_kernel<kMode, kA><<<(unsigned)P, Cfg<kMode>::kThreads, Cfg<kMode>::kSmem, st>>>(p);
  if (P > 1) {
    // programmatic dependent launch: the merge's blocks may be scheduled as the persistent CTAs
    // exit and wait (griddepcontrol.wait) for the whole grid's writes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P - 1), kBM / kCombineRows);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, prefill_combine_kernel, p);
  }
  return check_launch(name);
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
                                             const void* k16, int64_t max_ctx, void* out, void* workspace,
                                             int64_t workspace_bytes, int32_t* dev_err, void* stream) {
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
  PKV_ARG(!workspace || (aligned16(workspace) && workspace_bytes >= kCtaWsBytes),
          "paged_prefill_attn: workspace must be 16-byte aligned and hold at least %lld bytes (got %lld)",
          (long long)kCtaWsBytes, (long long)workspace_bytes);
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
  p.total_q = total_q;
  // block-aligned tiles where a 128-key tile could straddle two blocks of a request
  p.tpb = (block_size >= kBN && block_size % kBN != 0 && max_blocks > 1) ? (block_size + kBN - 1) / kBN : 0;
  p.tpb_inv = p.tpb ? 1.0f / (float)p.tpb : 0.0f;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.dev_err = dev_err;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int mode = !int8 ? 0 : (k16 ? 2 : 1);
  if (mode == 2) {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)num_kv_heads, (uint64_t)num_reqs * (uint64_t)max_ctx};
    const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)num_kv_heads * kD * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)kBN};
    pkv_status s = encode_tiled(&p.k16map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, k16, dims, strides, box, "k16");
    if (s != PKV_OK) return s;
  }
  const char* nm = "paged_prefill_attn";
  if (p.tpb) {
    if (mode == 0) return launch_prefill<0, true>(p, num_reqs, workspace, workspace_bytes, st, nm);
    if (mode == 1) return launch_prefill<1, true>(p, num_reqs, workspace, workspace_bytes, st, nm);
    return launch_prefill<2, true>(p, num_reqs, workspace, workspace_bytes, st, nm);
  }
  if (mode == 0) return launch_prefill<0, false>(p, num_reqs, workspace, workspace_bytes, st, nm);
  if (mode == 1) return launch_prefill<1, false>(p, num_reqs, workspace, workspace_bytes, st, nm);
  return launch_prefill<2, false>(p, num_reqs, workspace, workspace_bytes, st, nm);
}

extern "C" pkv_status pkv_paged_prefill_attn_fp8(const void* q, const uint8_t* k_fp8, const uint8_t* v_fp8,
                                                 const float* k_scale, const float* v_scale, int64_t num_blocks,
                                                 int64_t stride_blk, int64_t stride_tok, int64_t stride_head,
                                                 const int32_t* block_table, int64_t bt_stride, int32_t max_blocks,
                                                 const int32_t* seq_lens, const int32_t* query_start_loc,
                                                 int32_t num_reqs, int32_t total_q, int32_t max_q_len,
                                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t block_size, float softmax_scale, void* out,
                                                 void* workspace, int64_t workspace_bytes, int32_t* dev_err,
                                                 void* stream) {
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
  PKV_ARG(!workspace || (aligned16(workspace) && workspace_bytes >= kCtaWsBytes),
          "paged_prefill_attn_fp8: workspace must be 16-byte aligned and hold at least %lld bytes (got %lld)",
          (long long)kCtaWsBytes, (long long)workspace_bytes);

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
  p.total_q = total_q;
  // plain 128-key tiles: the converter warps read K/V rows one by one, so tiles that straddle
  // blocks cost nothing extra, and the tiles (so the arithmetic) are those of the dense-scratch path
  p.tpb = 0;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.dev_err = dev_err;
  p.k_fp8 = k_fp8;
  p.v_fp8 = v_fp8;
  p.stride_blk = stride_blk;
  p.stride_tok = stride_tok;
  p.stride_head = stride_head;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  return launch_prefill<3, false>(p, num_reqs, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                           "paged_prefill_attn_fp8");
}

extern "C" size_t pkv_paged_prefill_workspace_bytes(int32_t num_ctas) {
  return num_ctas > 0 ? (size_t)num_ctas * (size_t)pkv::kCtaWsBytes : 0;
}
