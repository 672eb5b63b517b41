// Block attention on the 5th-generation tensor cores (bf16 in, fp32 accumulate).
//
// Keys are taken as three contiguous ranges, each through its own TMA map so
// that no row outside a range is ever read: the cached prefix [0, f0), the fresh
// keys of this step (nq rows, the query positions) and the cached suffix
// [f1, N).  Softmax is invariant to the order of the keys, so the key tiles of
// 64 rows are enumerated range by range; with fewer fresh rows than a tile, the
// suffix's last, partial tile may complete the fresh one (a joined tile).
//
// One CTA = (sequence, KV head, 128-row query tile, split of the key tiles);
// all query heads sharing the KV head are packed into the 128 rows when
// nq <= 128.  Both operands that are reused across a tile's MMAs live in tensor
// memory, so the tensor core reads only K and V from shared memory:
//   TMEM   Q (128 rows x d bf16, written once), S0 / S1 (64 fp32 score columns
//          each), P0 / P1 (the probabilities as bf16 pairs), O0 / O1 (d fp32
//          columns each)
//   warp 0     TMA: the query tile once (into the last pipeline stage), then K
//              and V tiles into a ring of 7 stages (d = 128; 8 at d = 64), less
//              the one or two stages a split merge receives into
//   warps 1-2  MMA issuers, one per softmax group (warp 1 also owns TMEM):
//              S_i = Q K_i^T (M=128, N=64 keys, K=d, A from TMEM) and
//              O_g += P_i V_i (N=d, K=64 keys, P from TMEM, V read MN-major),
//              each issued as soon as its inputs are ready
//   warp 3     sends the split merge's rows to their owners
//   warps 4-7  softmax group 0: the even key tiles; warps 8-11 group 1: the odd
//              ones.  One thread per query row holds the tile's whole score row:
//              row max, lazy reference max (it moves only when a row's max
//              exceeds it by more than 2^8, and then O_g's row and l are
//              rescaled in TMEM after the group's previous PV product has
//              landed), P = 2^((S - m_ref) * scale * log2 e) stored as bf16 to
//              TMEM (after a group's first tile computed against the current
//              reference before the row max is known, and again if it moves).
//              Each group keeps its own (m, l, O_g); while one group
//              computes its softmax the tensor core works on the other's tile.
// At the end the two groups' rows are combined in the CTA.  Splits of one unit
// form a thread block cluster (<= 8) and merge through distributed shared
// memory.  Only the tile rows that can hold a query are merged (a DualCache
// tile of one MHA head has 32 such rows of 128); CTA c owns an equal share of
// them, [c R, (c + 1) R) in whole 8-row groups.  Every CTA stages its
// normalised copies of the rows it does not own in its own shared memory,
// grouped by owner, with each row's (max, sum), and sends each group to its
// owner with bulk copies that complete on the owner's mbarrier.  The owner
// receives them in ring stages the K/V pipeline leaves out, so no CTA waits for
// a peer's pipeline to finish before sending; it combines the C copies of its
// rows with weights 2^(m_c - M) L_c and writes them.
//
// K/V maps view [b, N, Hkv, d] as (d, position, head, b), so one box brings a
// tile half's keys of all heads packed in the tile, head-major.
//
// FP8 KV cache (F8KV): cached K and V are E4M3 codes with one power-of-two scale
// per (sequence, position, KV head) row.  A cache tile is loaded as bytes into
// the V half of its ring stage.  The softmax group that owns the tile turns its
// K codes into the bf16 K tile TMA would have written -- code * scale is exact
// in bf16 -- one of the group's tiles ahead (while it works on the previous
// one), which releases the tile to the group's MMA issuer, and its V codes into
// the bf16 V tile right after reading the tile's scores.  The products and the
// softmax arithmetic are unchanged.  Fresh K/V tiles are loaded as bf16
// directly.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 384;   // warps 0-3: TMA, two MMA issuers, merge sender; 4-11: two softmax groups
constexpr int kTile = 128;       // rows per query tile
constexpr int kKeys = 64;        // keys per key tile
constexpr int kMaxCluster = 8;   // portable thread-block cluster size
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMergeStages = 2;  // ring stages the split merge may take out of the K/V pipeline

struct Plan {
  int f0, f1;           // cached prefix [0, f0), cached suffix [f1, N)
  int ka, kf, kcn;      // key tiles in the three ranges
  int kt;               // total key tiles
  int nsplit;           // CTAs (cluster size) per unit
  int qr;               // query rows per head slot in a tile (multiple of 8)
  int ht;               // head slots per tile
  int qtiles_per_head;  // tiles per head when nq > 128 (0 when heads are packed)
  int nqt;              // query tiles per KV head group
  int kvp;              // KV heads per tile (1, or 2 / 4 for MHA with few queries)
  int tk;               // keys per KV head per key tile (64 / kvp)
  int abs_suffix;       // suffix rows are absolute cache rows (per-sequence blocks: full-cache maps)
  int units;            // batch * (Hkv / kvp) * nqt
  int nvr;              // tile rows that can hold a query (the rest are padding in every unit)
  int rpc;              // split merge: rows owned per CTA of a cluster (multiple of 8; 128 without a split)
  int nsp;              // ring stages of the K/V pipeline (the ring's last stages receive merged rows)
  // rows of the suffix's last, partial tile that share the one fresh tile (0: none).  With fewer fresh
  // rows than a tile, their tile is completed by the suffix's tail (rows [0, nq) fresh, [nq, nq + join)
  // the last cached rows), so the unit has one key tile less to split over its cluster.
  int join;
};

template <int D>
struct Cfg {
  static constexpr int DH = D / 64;                   // 64-column halves of a row
  static constexpr int QHALF = kTile * 128;           // 128 rows x 64 bf16
  static constexpr int KV_BYTES = kKeys * D * 2;      // 64 key rows x d bf16
  static constexpr int KVHALF = kKeys * 128;          // 64 rows x 64 bf16
  static constexpr int STAGE = 2 * KV_BYTES;          // K + V
  static constexpr int NS = D == 128 ? 7 : 8;         // K/V ring stages
  static_assert(kTile * D * 2 <= STAGE, "the query tile is staged in one ring stage");
  static constexpr int RING = NS * STAGE;
  // Split merge: a row sent to its owner is D fp32 values normalised by the row's sum (RB bytes), with
  // the row's (max in log2 units, sum) as a separate 8-byte pair.  The owner receives its peers' rows in
  // the ring's last stages, which the K/V pipeline then leaves out (at most kMergeStages), and their
  // pairs after the barriers (RECV_ML_BYTES).  Once the pipeline is done, its first stages hold the rows
  // this CTA sends (row r at r * RB) and their pairs, and the two groups' (max, sum) per row.
  static constexpr int RB = D * 4;                   // (16-byte chunk j of row r stored at chunk j ^ (r & 7))
  static constexpr int SEND_ML_OFF = kTile * RB;
  static constexpr int ML_OFF = (SEND_ML_OFF + kTile * 8 + 1023) / 1024 * 1024;
  static_assert(ML_OFF + 2 * kTile * 8 <= (NS - kMergeStages) * STAGE, "post-pipeline areas inside the pipeline");
  static constexpr int RECV_ML_BYTES = 1280;
  static constexpr int SMEM = RING + 1024 + 512 + RECV_ML_BYTES;    // + alignment + Bars + received pairs
  // TMEM columns
  static constexpr uint32_t Q_COL = 0;               // D / 2 columns of bf16 pairs
  static constexpr uint32_t S_COL = D / 2;           // S0, S1: 64 fp32 columns each
  static constexpr uint32_t P_COL = D / 2 + 128;     // P0, P1: 32 columns (64 bf16) each
  static constexpr uint32_t O_COL = D / 2 + 192;     // O0, O1: D fp32 columns each
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(O_COL + 2 * D <= TMEM_COLS, "TMEM budget");
};

struct Bars {
  uint64_t qfull, qtmem, kvfull[8], kvempty[8], raw[8], sfull[2], sempty[2], pfull[2], pvdone[2], drain, mrg;
  uint32_t tmem_base;
  int32_t abort;
  int32_t issued;     // K/V tiles issued by the producer
  int32_t consumed_g[2];   // per group: key tiles whose arrival its MMA issuer waited for
};

// The two softmax warps of TMEM lane quadrant q (warps 4 + q and 8 + q) synchronise as a pair.
__device__ __forceinline__ void quadrant_bar(int q) { asm volatile("bar.sync %0, 64;" ::"r"(2 + q) : "memory"); }
// The four warps of softmax group g.
__device__ __forceinline__ void group_bar(int g) { asm volatile("bar.sync %0, 128;" ::"r"(7 + g) : "memory"); }
// The softmax warps and warp 3, which sends the split merge's rows once the softmax warps have staged them.
__device__ __forceinline__ void send_bar() { asm volatile("bar.sync 9, 288;" ::: "memory"); }

// The maximum of m[0, LEN) by three-input maxima, level by level in place (LEN / 2 instructions for LEN
// a power of two): every index is known at compile time, so the array stays in registers.
template <int LEN, int CAP>
struct Max3Tree {
  static __device__ __forceinline__ float run(float (&m)[CAP]) {
    constexpr int OUT = (LEN + 2) / 3;
#pragma unroll
    for (int e = 0; e < OUT; ++e) {
      if (3 * e + 2 < LEN) m[e] = tc::max3(m[3 * e], m[3 * e + 1], m[3 * e + 2]);
      else if (3 * e + 1 < LEN) m[e] = fmaxf(m[3 * e], m[3 * e + 1]);
      else m[e] = m[3 * e];
    }
    return Max3Tree<OUT, CAP>::run(m);
  }
};
template <int CAP>
struct Max3Tree<1, CAP> {
  static __device__ __forceinline__ float run(float (&m)[CAP]) { return m[0]; }
};

struct KeyTile {
  int range;   // 0 prefix cache, 1 fresh, 2 suffix cache
  int row0;    // first row within the range's map
  int nvalid;  // valid keys in the tile (per KV head)
};

__device__ __forceinline__ KeyTile key_tile(const Plan &pl, int nq, int n, int k) {
  KeyTile t;
  if (k < pl.ka) {
    t.range = 0; t.row0 = k * pl.tk; t.nvalid = min(pl.tk, pl.f0 - t.row0);
  } else if (k < pl.ka + pl.kf) {
    t.range = 1; t.row0 = (k - pl.ka) * pl.tk; t.nvalid = min(pl.tk, nq - t.row0) + pl.join;
  } else {
    const int r2 = (k - pl.ka - pl.kf) * pl.tk;    // row within the suffix
    t.range = 2; t.row0 = (pl.abs_suffix ? pl.f1 : 0) + r2; t.nvalid = min(pl.tk, n - pl.f1 - r2);
  }
  return t;
}

struct Args {
  Plan pl;
  int batch, n, nq, hq, hkv, group;
  float scale_log2;  // softmax scale * log2(e)
  float scale;
  int out_f32;
  void *out;
  float *lse;
  int32_t *err;
  const int32_t *blocks;   // per-sequence DualCache block indices (null: the plan's window for all)
  int prompt_len, nblocks;
  const float *k_scale, *v_scale;   // F8KV: scales of the cached rows [b, N, Hkv]
  // cache update fused into the call: the first `win` fresh rows (the block) are stored into cache rows
  // [f0, f0 + win) of each sequence by the CTAs that load them (those of the KV head group's first query
  // tile), in boxes of `win_box` rows (0: no update)
  int win, win_box;
};

// 4 E4M3 codes (one 32-bit word) times `sc` as 4 bf16 (two words); exact: an E4M3 value has at most
// 4 significant bits and `sc` is a power of two.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w, float sc) {
  uint32_t o[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> (16 * h)), __NV_E4M3);
    const float2 f = __half22float2(*(const __half2 *)&hr);
    const float2 g = tc::f2_unpack(tc::f2_mul(tc::f2_pack(f.x, f.y), tc::f2_pack(sc, sc)));   // both lanes at once
    const __nv_bfloat162 b = __floats2bfloat162_rn(g.x, g.y);
    o[h] = *(const uint32_t *)&b;
  }
  return make_uint2(o[0], o[1]);
}

// Rotation of the code chunks of half h of row r: a quarter warp (four rows, both halves) then reads its
// codes and writes its bf16 chunks in eight distinct 16-byte bank groups.
template <int D>
__device__ __forceinline__ int half_rot(int r, int h) { return D == 128 ? r + 2 * h : (r >> 1) + h; }

// The D / 2 codes of half h of row r (D / 32 chunks of 16), slot c holding chunk (c + half_rot) mod D / 32.
template <int D>
__device__ __forceinline__ void load_code_half(const unsigned char *half, int r, int h, uint4 (&codes)[D / 32]) {
  constexpr int NC = D / 32;
  const int rot = half_rot<D>(r, h);
#pragma unroll
  for (int c = 0; c < NC; ++c) codes[c] = *(const uint4 *)(half + ((c + rot) & (NC - 1)) * 16);
}

// Half h of row r of a bf16 K or V tile in the layout the 128-byte-swizzled TMA load writes (64-column
// halves of kKeys rows x 128 bytes, 16-byte chunk j of row r at chunk j ^ (r & 7); d = 128: half h is the
// whole row of 64-column half h, d = 64: chunks [4 h, 4 h + 4) of the single row): sc x the codes that
// load_code_half read, or zeros where !valid (not code x 0, which is NaN for a NaN code).
template <int D>
__device__ __forceinline__ void store_bf16_half(unsigned char *tile, int r, int h, const uint4 (&codes)[D / 32],
                                                float sc, bool valid) {
  constexpr int NC = D / 32;
  unsigned char *row = tile + (D == 128 ? h * (kKeys * 128) : 0) + r * 128;
  const int j0 = D == 128 ? 0 : 4 * h;
  const int rot = half_rot<D>(r, h);
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int j = j0 + 2 * ((c + rot) & (NC - 1));
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
    if (valid) {
      const uint2 x0 = e4m3x4_to_bf16x4(codes[c].x, sc), x1 = e4m3x4_to_bf16x4(codes[c].y, sc);
      const uint2 x2 = e4m3x4_to_bf16x4(codes[c].z, sc), x3 = e4m3x4_to_bf16x4(codes[c].w, sc);
      lo = make_uint4(x0.x, x0.y, x1.x, x1.y);
      hi = make_uint4(x2.x, x2.y, x3.x, x3.y);
    }
    *(uint4 *)(row + ((j ^ (r & 7)) * 16)) = lo;
    *(uint4 *)(row + (((j + 1) ^ (r & 7)) * 16)) = hi;
  }
}

// Scale of key row r (KV head kvh + r / tk, key r % tk) of cache tile t: the key's cache position is
// absolute for prefix rows, relative to f1 for suffix rows unless the maps cover the whole cache;
// rows past N were zero-filled and get scale 0.
__device__ __forceinline__ float cache_scale(const Args &a, const Plan &pl, const KeyTile &t, int b, int kvh, int r,
                                             const float *scale) {
  const int hp = r / pl.tk;
  const int pos = (t.range == 2 && !pl.abs_suffix ? pl.f1 : 0) + t.row0 + (r - hp * pl.tk);
  return pos < a.n ? __ldg(scale + ((int64_t)b * a.n + pos) * a.hkv + kvh + hp) : 0.f;
}

__device__ __forceinline__ void fail(Bars &br, int32_t *err, int site) {
  record_device_error(err, site);
  atomicExch(&br.abort, 1);
}

// Output row of the query tile -> (head slot, query index); false if padding.
__device__ __forceinline__ bool row_target(const Plan &pl, int nq, int nh, int q0, int r, int &hs, int &qi) {
  hs = pl.qtiles_per_head == 0 ? r / pl.qr : 0;
  qi = pl.qtiles_per_head == 0 ? r % pl.qr : q0 + r;
  return hs < nh && qi < nq;
}

// D / 2 values as bf16 (8 per 16-byte chunk) or fp32 (4 per chunk) at `dst`.
template <int N>
__device__ __forceinline__ void store_row_part(void *dst, bool f32, const float (&v)[N], float inv) {
  if (f32) {
    float4 *o = (float4 *)dst;
#pragma unroll
    for (int c = 0; c < N / 4; ++c) o[c] = make_float4(v[4 * c] * inv, v[4 * c + 1] * inv, v[4 * c + 2] * inv, v[4 * c + 3] * inv);
  } else {
    uint4 *o = (uint4 *)dst;
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * c + 2 * e] * inv, v[8 * c + 2 * e + 1] * inv);
        w[e] = *(uint32_t *)&h2;
      }
      o[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

static_assert(sizeof(Bars) <= 512, "Bars must fit its shared-memory reservation");

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

template <int D, int KVP, bool F8KV>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mka,
                   const __grid_constant__ CUtensorMap mkf, const __grid_constant__ CUtensorMap mkc,
                   const __grid_constant__ CUtensorMap mva, const __grid_constant__ CUtensorMap mvf,
                   const __grid_constant__ CUtensorMap mvc,
                   const __grid_constant__ CUtensorMap mwk, const __grid_constant__ CUtensorMap mwv,
                   const __grid_constant__ CUtensorMap mkt, const __grid_constant__ CUtensorMap mvt, const Args a) {
  using CF = Cfg<D>;
  constexpr int NS = CF::NS;
  constexpr int TK = kKeys / KVP;                      // keys of one KV head in a key tile
  extern __shared__ unsigned char smem_raw[];
  unsigned char *kv_s = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);   // NS stages
  Bars &br = *(Bars *)(kv_s + CF::RING);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Plan pl = a.pl;   // per-sequence blocks fill in this CTA's ranges after the dependency wait
  const int ns = pl.nsp;                               // K/V pipeline stages
  // the query tile, until it is in TMEM: in the first receive stage of a split merge (no peer sends
  // before every CTA of the cluster has moved its query tile out, see below), else in the last stage
  unsigned char *q_s = kv_s + (pl.nsplit > 1 ? ns : ns - 1) * CF::STAGE;

  const int split = blockIdx.x % pl.nsplit;
  const int unit = blockIdx.x / pl.nsplit;
  const int nkvg = a.hkv / KVP;                        // KV head groups
  const int qt = unit % pl.nqt;
  const int kvh = ((unit / pl.nqt) % nkvg) * KVP;      // first KV head of this tile
  const int b = unit / (pl.nqt * nkvg);
  int h0, nh, q0;
  if (KVP > 1) {
    h0 = 0; nh = KVP; q0 = 0;                          // head slot s = KV head kvh + s (MHA)
  } else if (pl.qtiles_per_head == 0) {
    h0 = qt * pl.ht; nh = min(pl.ht, a.group - h0); q0 = 0;
  } else {
    h0 = qt / pl.qtiles_per_head; nh = 1; q0 = (qt % pl.qtiles_per_head) * kTile;
  }
  const int C = pl.nsplit;                             // CTAs of this unit's cluster
  const int rpc = pl.rpc;                              // rows owned per CTA in the split merge
  const int crank = C > 1 ? (int)tc::cluster_ctarank() : 0;
  // rows of owner c that are merged: its share of the rows that can hold a query
  auto seg_rows = [&](int c) { return max(0, min(rpc, pl.nvr - c * rpc)); };

  if (threadIdx.x == 0) {
    br.abort = 0; br.issued = 0; br.consumed_g[0] = 0; br.consumed_g[1] = 0;
    tc::mbar_init(&br.qfull, 1);
    tc::mbar_init(&br.qtmem, 4);
    for (int i = 0; i < NS; ++i) {
      tc::mbar_init(&br.kvfull[i], 1);
      tc::mbar_init(&br.kvempty[i], 1);
      tc::mbar_init(&br.raw[i], 1);
    }
    for (int g = 0; g < 2; ++g) {
      tc::mbar_init(&br.sfull[g], 1);
      tc::mbar_init(&br.sempty[g], 4);
      tc::mbar_init(&br.pfull[g], 4);
      tc::mbar_init(&br.pvdone[g], 1);
    }
    tc::mbar_init(&br.drain, 2);                     // one arrival per MMA issuer
    tc::mbar_init(&br.mrg, 1);
    tc::fence_barrier_init();
    // the merge barrier expects the other C - 1 CTAs' copies of this one's rows and their pairs
    if (C > 1) tc::mbar_arrive_expect_tx(&br.mrg, (uint32_t)((C - 1) * seg_rows(crank) * (CF::RB + 8)));
    for (const CUtensorMap *m : {&mq, &mka, &mkf, &mkc, &mva, &mvf, &mvc}) tc::prefetch_tensormap(m);
    if (a.win_box > 0) { tc::prefetch_tensormap(&mwk); tc::prefetch_tensormap(&mwv); }
    if (pl.join > 0) { tc::prefetch_tensormap(&mkt); tc::prefetch_tensormap(&mvt); }
  }
  if (warp == 1) tc::tmem_alloc(&br.tmem_base, CF::TMEM_COLS);
  // Launched as a programmatic dependent: everything above overlaps the previous kernel in the
  // stream, which may produce q, the caches or the fresh K/V (or still read the output).
  tc::pdl_wait_primary();
  tc::pdl_launch_dependents();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = br.tmem_base;
  if (a.blocks != nullptr) {
    // this sequence's own block: cached prefix [0, f0), fresh window [f0, f1), cached suffix [f1, N);
    // an index outside [0, nblocks) gives no key tiles (and device error 232)
    const int bi = a.blocks[b];
    if (bi >= 0 && bi < a.nblocks) {
      pl.f0 = a.prompt_len + bi * a.nq;
      pl.f1 = pl.f0 + a.nq;
      pl.ka = (pl.f0 + pl.tk - 1) / pl.tk;
      pl.kf = (a.nq + pl.tk - 1) / pl.tk;
      pl.kcn = (a.n - pl.f1 + pl.tk - 1) / pl.tk;
      pl.kt = pl.ka + pl.kf + pl.kcn;
    } else {
      pl.kt = 0;
      if (threadIdx.x == 0 && split == 0) record_device_error(a.err, 232);
    }
  }
  const int k0 = (int)((int64_t)pl.kt * split / pl.nsplit);
  const int nt = (int)((int64_t)pl.kt * (split + 1) / pl.nsplit) - k0;
  // set by the first wait that gives up (fail()); every later wait that polls it returns at once
  const volatile int32_t *abort_flag = &br.abort;

  // thread of the softmax groups: its query row, group and running state
  const int g = (warp - 4) >> 2;                       // softmax group (warps >= 4)
  const int r = (warp & 3) * 32 + lane;
  float m_run = kNegInf, l_run = 0.f;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const uint64_t pol_q = tc::policy_evict_last();
      const uint64_t pol_kv = tc::policy_evict_first();
      tc::mbar_arrive_expect_tx(&br.qfull, (uint32_t)(pl.qr * 128 * CF::DH * nh));
      for (int hs = 0; hs < nh; ++hs)
        for (int dh = 0; dh < CF::DH; ++dh)
          tc::tma_load_4d(q_s + dh * CF::QHALF + hs * pl.qr * 128, &mq, &br.qfull, dh * 64,
                          kvh * a.group + h0 + hs, q0, b, pol_q);
      int st = 0;                                      // tile i's ring stage and that stage's phase parity
      uint32_t ph = 0;
      for (int i = 0; i < nt && !*abort_flag; ++i, st = st + 1 == ns ? 0 : st + 1, ph ^= st == 0 ? 1u : 0u) {
        // without a cluster the last stage holds the query tile until group 0 has copied it into TMEM
        if (C == 1 && i == ns - 1 && !tc::mbar_wait_or_abort(&br.qtmem, 0, abort_flag)) {
          if (!*abort_flag) fail(br, a.err, 210);
          break;
        }
        if (!tc::mbar_wait_or_abort(&br.kvempty[st], ph ^ 1u, abort_flag)) {
          if (!*abort_flag) fail(br, a.err, 211);
          break;
        }
        const KeyTile kt = key_tile(pl, a.nq, a.n, k0 + i);
        const CUtensorMap *mk = kt.range == 0 ? &mka : (kt.range == 1 ? &mkf : &mkc);
        const CUtensorMap *mv = kt.range == 0 ? &mva : (kt.range == 1 ? &mvf : &mvc);
        unsigned char *ks = kv_s + st * CF::STAGE;
        if (F8KV && kt.range != 1) {
          // cache tile: K codes then V codes (kKeys rows x D bytes each) into the stage's V half; the
          // tile's softmax group writes the bf16 tiles (the K tile completes kvfull)
          tc::mbar_arrive_expect_tx(&br.raw[st], (uint32_t)(2 * kKeys * D));
          // one box: kKeys / KVP keys of each of the KVP heads, head-major
          tc::tma_load_4d(ks + CF::KV_BYTES, mk, &br.raw[st], 0, kt.row0, kvh, b, pol_kv);
          tc::tma_load_4d(ks + CF::KV_BYTES + kKeys * D, mv, &br.raw[st], 0, kt.row0, kvh, b, pol_kv);
        } else {
          tc::mbar_arrive_expect_tx(&br.kvfull[st], (uint32_t)CF::STAGE);
          for (int dh = 0; dh < CF::DH; ++dh) {   // per 64-column half, the tile's 64 key rows: KVP heads x
            const int off = dh * CF::KVHALF;        // (64 / KVP) keys, head-major, in one box
            tc::tma_load_4d(ks + off, mk, &br.kvfull[st], dh * 64, kt.row0, kvh, b, pol_kv);
            tc::tma_load_4d(ks + CF::KV_BYTES + off, mv, &br.kvfull[st], dh * 64, kt.row0, kvh, b, pol_kv);
            if (kt.range == 1 && pl.join > 0) {
              // the joined tile: the nq fresh rows (a box of nq rows) then the suffix's tail (a box of the
              // remaining tk - nq rows from its last, partial tile; rows past the cache read as zeros)
              const int ro = a.nq * 128;           // a multiple of 1024 bytes: the swizzle atoms line up
              tc::tma_load_4d(ks + off + ro, &mkt, &br.kvfull[st], dh * 64, pl.kcn * pl.tk, kvh, b, pol_kv);
              tc::tma_load_4d(ks + CF::KV_BYTES + off + ro, &mvt, &br.kvfull[st], dh * 64, pl.kcn * pl.tk, kvh, b,
                              pol_kv);
            }
          }
        }
        atomicExch(&br.issued, i + 1);
      }
    }
  } else if (warp == 1 || warp == 2) {
    if (lane == 0) {
      // ---------------- MMA issuers, one per softmax group ----------------
      // Warp 1 serves group 0 (the even key tiles), warp 2 group 1 (the odd ones).  Each issues its
      // group's S_j = Q K_j^T as soon as the tile has landed and the group has read S_{j-2} from its
      // score buffer, and O_g += P_i V_i as soon as the group has stored P_i, whichever is ready first
      // (a PV first when both are), so the two groups' products never wait on each other's issue.
      const int gg = warp - 1;
      const uint32_t id_s = tc::idesc_bf16_f32(128, kKeys, 0);
      const uint32_t id_o = tc::idesc_bf16_f32(128, D, 1);
      bool run = tc::mbar_wait_or_abort(&br.qtmem, 0, abort_flag);    // Q is in TMEM
      if (!run && !*abort_flag) fail(br, a.err, 212);
      int js = gg, jp = gg;                             // next S, next PV of this group
      int js_st = gg, jp_st = gg;                       // their ring stages
      uint32_t js_ph = 0;                               // phase parity of js's stage
      // this CTA stores the block's fresh K/V into the cache window when the call asks for it and it
      // serves the first query tile of its KV head group (every such CTA of the split covers its own keys)
      const bool update_cache = a.win_box > 0 && qt == 0;
      bool stored_pending = false;
      uint64_t t0 = tc::globaltimer();
      for (uint32_t spin = 0; run && jp < nt; ++spin) {
        if (jp < js && tc::mbar_test_wait(&br.pfull[gg], (uint32_t)(jp >> 1) & 1u)) {
          const int st = jp_st;
          tc::fence_after_sync();
          const uint32_t va = tc::smem_u32(kv_s + st * CF::STAGE + CF::KV_BYTES);
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks)
            tc::mma_bf16_ts(tmem + CF::O_COL + (uint32_t)(gg * D), tmem + CF::P_COL + (uint32_t)(gg * 32 + ks * 8),
                            tc::sw128_mn_desc(va + (uint32_t)(ks * 2048), CF::KVHALF), id_o, (jp >= 2) || ks != 0);
          tc::mma_commit(&br.pvdone[gg]);
          if (stored_pending) {                         // the cache-window stores have read the stage
            tc::bulk_wait_read_all();
            stored_pending = false;
          }
          tc::mma_commit(&br.kvempty[st]);
          jp += 2;
          jp_st += 2;
          if (jp_st >= ns) jp_st -= ns;
          t0 = tc::globaltimer();
          continue;
        }
        if (js < nt && tc::mbar_test_wait(&br.kvfull[js_st], js_ph) &&
            tc::mbar_test_wait(&br.sempty[gg], ((uint32_t)(js >> 1) & 1u) ^ 1u)) {
          const int st = js_st;
          tc::fence_after_sync();
          const uint32_t ka = tc::smem_u32(kv_s + st * CF::STAGE);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            tc::mma_bf16_ts(tmem + CF::S_COL + (uint32_t)(gg * kKeys), tmem + CF::Q_COL + (uint32_t)(ks * 8),
                            tc::sw128_desc(ka + (ks / 4) * CF::KVHALF + (uint32_t)((ks % 4) * 32)), id_s, ks != 0);
          tc::mma_commit(&br.sfull[gg]);
          if (update_cache) {
            // the block's fresh rows of this tile into the cache window (rows past the block lie outside
            // the box); the stage is released only after the stores have read it (wait below)
            const KeyTile kt = key_tile(pl, a.nq, a.n, k0 + js);
            if (kt.range == 1 && kt.row0 < a.win) {
              unsigned char *ks_ = kv_s + st * CF::STAGE;
              for (int dh = 0; dh < CF::DH; ++dh) {
                tc::tma_store_4d(&mwk, ks_ + dh * CF::KVHALF, dh * 64, pl.f0 + kt.row0, kvh, b);
                tc::tma_store_4d(&mwv, ks_ + CF::KV_BYTES + dh * CF::KVHALF, dh * 64, pl.f0 + kt.row0, kvh, b);
              }
              tc::bulk_commit_group();
              stored_pending = true;
            }
          }
          js += 2;
          js_st += 2;
          if (js_st >= ns) { js_st -= ns; js_ph ^= 1u; }
          atomicExch(&br.consumed_g[gg], js >> 1);
          t0 = tc::globaltimer();
          continue;
        }
        if ((spin & 63u) == 0) {
          if (*abort_flag) break;
          if (tc::globaltimer() - t0 > tc::kWaitLimitNs) {
            fail(br, a.err, jp < js ? 215 : 213);
            break;
          }
        }
      }
      if (update_cache) tc::bulk_wait_read_all();      // the window stores have read the ring
      tc::mma_commit(&br.drain);                        // both issuers arrive: count 2
      if (!tc::mbar_wait(&br.drain, 0)) record_device_error(a.err, 217);
    }
  } else if (warp >= 4) {
    // Every softmax warp runs every tile of its group and meets every named barrier the same number of
    // times, whatever its waits return: a wait that gives up only marks this thread's result invalid
    // (ok = false), records the site and raises the abort flag, after which every wait of the CTA
    // returns at once.  So no warp can be left waiting at a named barrier for a partner that has left.
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int gt = threadIdx.x - 128 - 128 * g;        // thread index within the group
    const int slot = KVP > 1 ? r / pl.qr : 0;         // KVP > 1: this row's head slot (uniform per warp)
    const uint32_t s_col = tmem + lane_base + CF::S_COL + (uint32_t)(g * kKeys + slot * TK);
    const uint32_t p_col = tmem + lane_base + CF::P_COL + (uint32_t)(g * 32);
    const uint32_t o_col = tmem + lane_base + CF::O_COL + (uint32_t)(g * D);
    if (g == 0) {
      // the query tile into TMEM: row r as D / 2 columns of bf16 pairs (rows of absent head slots: zeros)
      if (!tc::mbar_wait_or_abort(&br.qfull, 0, abort_flag)) {
        if (!*abort_flag) fail(br, a.err, 216);
        ok = false;
      }
      const bool qvalid = pl.qtiles_per_head != 0 || r < nh * pl.qr;
#pragma unroll
      for (int dh = 0; dh < CF::DH; ++dh) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = qvalid ? *(const uint4 *)(q_s + dh * CF::QHALF + r * 128 + ((c ^ (r & 7)) * 16))
                                 : make_uint4(0u, 0u, 0u, 0u);
          w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
        tc::tmem_st_32x32b_x32(tmem + lane_base + CF::Q_COL + (uint32_t)(dh * 32), w);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&br.qtmem);
    }
    // the query tile has left the receive stage (its loads are complete: their values are in TMEM)
    if (C > 1 && g == 0) tc::cluster_arrive_relaxed();
    if (KVP > 1) {
      // each row writes only its head's block of P: the rest of its P row stays zero
      uint32_t z[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) z[e] = 0u;
      tc::tmem_st_32x32b_x32(p_col, z);
      tc::tmem_st_wait();
    }
    const float sl2 = a.scale_log2;
    // F8KV: the group converts its cache tiles' K rows one of its tiles ahead (tile i + 2 while it works on
    // tile i, its first before the loop) and their V rows at the tile itself; thread gt handles half hh of
    // key row kr of both.  rawpar: the raw barriers' phase parities (bit st: cache tiles loaded into stage
    // st so far), advanced over every tile before the one whose codes are awaited.
    const int kr = gt >> 1, hh = gt & 1;
    uint32_t rawpar = 0;
    int seen = 0, seen_st = 0;
    auto scale_of = [&](int j, const float *sc) -> float {   // row kr's scale in tile j (0: none)
      if (!F8KV || j >= nt) return 0.f;
      const KeyTile t = key_tile(pl, a.nq, a.n, k0 + j);
      if (t.range == 1 || (kr % pl.tk) >= t.nvalid) return 0.f;
      return cache_scale(a, pl, t, b, kvh, kr, sc);
    };
    auto convert_k = [&](int j, int stj, float ksc) {        // cache tile j's K rows; completes kvfull
      for (; seen < j; ++seen, seen_st = seen_st + 1 == ns ? 0 : seen_st + 1)
        if (key_tile(pl, a.nq, a.n, k0 + seen).range != 1) rawpar ^= 1u << seen_st;
      const bool got = tc::mbar_wait_or_abort(&br.raw[stj], (rawpar >> stj) & 1u, abort_flag);
      if (!got) {
        if (!*abort_flag) fail(br, a.err, 220);
        ok = false;
      }
      unsigned char *sj = kv_s + stj * CF::STAGE;
      uint4 kc[D / 32];
      load_code_half<D>(sj + CF::KV_BYTES + kr * D + hh * (D / 2), kr, hh, kc);
      store_bf16_half<D>(sj, kr, hh, kc, ksc, (kr % pl.tk) < key_tile(pl, a.nq, a.n, k0 + j).nvalid);
      tc::fence_proxy_async_smem();
      group_bar(g);                                    // every K row of the tile is written
      if (gt == 0 && got) tc::mbar_arrive(&br.kvfull[stj]);
    };
    float ksc_n = scale_of(g + 2, a.k_scale);          // K scale of the tile converted in the next iteration
    float vsc_n = scale_of(g, a.v_scale);              // V scale of the next iteration's tile
    if (F8KV && g < nt && key_tile(pl, a.nq, a.n, k0 + g).range != 1) convert_k(g, g, scale_of(g, a.k_scale));
    int u = 0;                                         // this group's tile count
    int st = g;                                        // tile i's ring stage
    for (int i = g; i < nt; i += 2, ++u, st = st + 2 >= ns ? st + 2 - ns : st + 2) {
      const KeyTile kt = key_tile(pl, a.nq, a.n, k0 + i);
      const float ksc2 = ksc_n, vsc = vsc_n;
      if constexpr (F8KV) {                            // loaded one iteration ahead of their use
        ksc_n = scale_of(i + 4, a.k_scale);
        vsc_n = scale_of(i + 2, a.v_scale);
      }
      const int nv = kt.nvalid;
      if (!tc::mbar_wait_or_abort(&br.sfull[g], (uint32_t)u & 1u, abort_flag)) {
        if (!*abort_flag) fail(br, a.err, 218);
        ok = false;
      }
      tc::fence_after_sync();
      // bf16 cache, per-sequence blocks: zeros over the tile's V rows outside the sequence's key range
      // (window rows at the edge of the prefix, which must not reach the product even as 0 * inf)
      if (!F8KV && a.blocks != nullptr && kt.range == 0 && nv < pl.tk) {
        if ((kr % pl.tk) >= nv) {
          unsigned char *row = kv_s + st * CF::STAGE + CF::KV_BYTES + (D == 128 ? hh * CF::KVHALF : 0) + kr * 128;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            const int j = (D == 128 ? 0 : 4 * hh) + c;
            *(uint4 *)(row + ((j ^ (kr & 7)) * 16)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        tc::fence_proxy_async_smem();
      }
      float x[TK];
      {
        uint32_t xr[TK];
        if constexpr (TK == 64) {
          tc::tmem_ld_32x32b_x32(s_col, *(uint32_t(*)[32])&xr[0]);
          tc::tmem_ld_32x32b_x32(s_col + 32, *(uint32_t(*)[32])&xr[32]);
        } else if constexpr (TK == 32) {
          tc::tmem_ld_32x32b_x32(s_col, xr);
        } else {
          tc::tmem_ld_32x32b_x16(s_col, xr);
        }
        tc::tmem_ld_wait();
        if (nv >= TK) {                                // a full tile: no per-key validity test
#pragma unroll
          for (int e = 0; e < TK; ++e) x[e] = __uint_as_float(xr[e]);
        } else {
#pragma unroll
          for (int e = 0; e < TK; ++e) x[e] = e < nv ? __uint_as_float(xr[e]) : kNegInf;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&br.sempty[g]);  // S_g may be overwritten by this group's next S
      if constexpr (F8KV) {
        // the K rows of this group's next tile (its score product may then start), and this tile's V rows:
        // their codes landed with its K codes (waited for then); they are read before the barrier, as the
        // bf16 V tile is written over them
        const int st2 = st + 2 >= ns ? st + 2 - ns : st + 2;
        if (i + 2 < nt && key_tile(pl, a.nq, a.n, k0 + i + 2).range != 1) convert_k(i + 2, st2, ksc2);
        if (kt.range != 1) {
          unsigned char *vt = kv_s + st * CF::STAGE + CF::KV_BYTES;
          uint4 vc[D / 32];
          load_code_half<D>(vt + kKeys * D + kr * D + hh * (D / 2), kr, hh, vc);
          group_bar(g);                                // every V code of the tile has been read
          store_bf16_half<D>(vt, kr, hh, vc, vsc, (kr % pl.tk) < nv);
          tc::fence_proxy_async_smem();
        }
      }
      // P = 2^(S scale log2(e) - ms) into pw (bf16 pairs) and its four partial row sums into lt
      uint32_t pw[TK / 2];
      float lt[4];
      auto exps = [&](float ms) {
        if (nv >= TK) {
          // key pairs: one paired fma for both exponents' arguments, one paired add into two running sums
          const uint64_t sc2 = tc::f2_pack(sl2, sl2), ms2 = tc::f2_pack(-ms, -ms);
          uint64_t acc[2] = {tc::f2_pack(0.f, 0.f), tc::f2_pack(0.f, 0.f)};
#pragma unroll
          for (int e = 0; e < TK / 2; ++e) {
            const float2 ar = tc::f2_unpack(tc::f2_fma(tc::f2_pack(x[2 * e], x[2 * e + 1]), sc2, ms2));
            const float p0 = tc::ex2_approx(ar.x), p1 = tc::ex2_approx(ar.y);
            acc[e & 1] = tc::f2_add(acc[e & 1], tc::f2_pack(p0, p1));
            __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
            pw[e] = *(uint32_t *)&h2;
          }
          const float2 s0 = tc::f2_unpack(acc[0]), s1 = tc::f2_unpack(acc[1]);
          lt[0] = s0.x; lt[1] = s0.y; lt[2] = s1.x; lt[3] = s1.y;
        } else {
          lt[0] = lt[1] = lt[2] = lt[3] = 0.f;
#pragma unroll
          for (int e = 0; e < TK / 2; ++e) {
            const float p0 = 2 * e < nv ? tc::ex2_approx(fmaf(x[2 * e], sl2, -ms)) : 0.f;
            const float p1 = 2 * e + 1 < nv ? tc::ex2_approx(fmaf(x[2 * e + 1], sl2, -ms)) : 0.f;
            lt[e & 3] += p0 + p1;
            __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
            pw[e] = *(uint32_t *)&h2;
          }
        }
      };
      // After the first tile the reference max rarely moves, so P is computed against it at once, beside
      // the row max (three-input maxima: a tree of TK / 2 instructions), and before the wait for the
      // previous PV product, which only the store of P and a rescale need; a tile whose max does move
      // the reference is computed again below.
      if (u > 0) exps(m_run * sl2);
      float mx[TK];
#pragma unroll
      for (int e = 0; e < TK; ++e) mx[e] = x[e];
      const float tm = Max3Tree<TK, TK>::run(mx);
      // the group's previous PV product has read P_g and finished updating O_g
      if (u > 0 && !tc::mbar_wait_or_abort(&br.pvdone[g], (uint32_t)(u - 1) & 1u, abort_flag)) {
        if (!*abort_flag) fail(br, a.err, 219);
        ok = false;
      }
      tc::fence_after_sync();
      const bool need = m_run == kNegInf || (tm - m_run) * sl2 > 8.f;
      if (u == 0 || __any_sync(0xffffffffu, need)) {
        const float m_new = need ? fmaxf(m_run, tm) : m_run;
        const float al = tc::ex2_approx((m_run - m_new) * sl2);   // 0 on a row's first tile
        if (u > 0) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc::tmem_ld_32x32b_x32(o_col + (uint32_t)c0, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * al);
            tc::tmem_st_32x32b_x32(o_col + (uint32_t)c0, o);
          }
        }
        l_run *= al;
        m_run = m_new;
        exps(m_run * sl2);
      }
      l_run += (lt[0] + lt[1]) + (lt[2] + lt[3]);
      if constexpr (TK == 64) tc::tmem_st_32x32b_x32(p_col, *(const uint32_t(*)[32])&pw[0]);
      else if constexpr (TK == 32) tc::tmem_st_32x32b_x16(p_col + (uint32_t)(slot * (TK / 2)), pw);
      else tc::tmem_st_32x32b_x8(p_col + (uint32_t)(slot * (TK / 2)), pw);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&br.pfull[g]);
    }
    // O_g is complete once the group's last PV product has landed
    if (u > 0 && !tc::mbar_wait_or_abort(&br.pvdone[g], (uint32_t)(u - 1) & 1u, abort_flag)) {
      if (!*abort_flag) fail(br, a.err, 219);
      ok = false;
    }
    tc::fence_after_sync();
  }

  // ---- every role is done: all copies consumed, all MMAs complete ----
  // With a cluster, the first cluster barrier says that this CTA's merge barrier is initialised and its
  // receive stage free: softmax group 0 arrived once the query tile was in TMEM, the other warps arrive
  // here.  Every CTA waits for it before its first copy to a peer.
  if (C > 1 && (warp < 4 || warp >= 8)) tc::cluster_arrive_relaxed();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      // copies issued but never consumed still land in shared memory: wait for them (bounded)
      tc::mbar_wait(&br.qfull, 0);
      for (int i = 0; i < br.issued; ++i) {
        if ((i >> 1) < br.consumed_g[i & 1]) continue;
        if (F8KV && key_tile(pl, a.nq, a.n, k0 + i).range != 1) {
          int uses = 0;                                // earlier cache tiles in this stage: raw's phase
          for (int j = i % ns; j < i; j += ns) uses += key_tile(pl, a.nq, a.n, k0 + j).range != 1;
          tc::mbar_wait(&br.raw[i % ns], (uint32_t)uses & 1u);
        } else {
          tc::mbar_wait(&br.kvfull[i % ns], (uint32_t)(i / ns) & 1u);
        }
      }
    }
    __syncthreads();
  }

  // ---- combine the two groups' rows: row r's final (M, L) and D values ----
  unsigned char *send = kv_s;                           // rows sent to their owners (row r at r * RB)
  float2 *send_ml = (float2 *)(kv_s + CF::SEND_ML_OFF);
  unsigned char *recv = kv_s + ns * CF::STAGE;          // peers' copies of the owned rows, by peer slot
  float2 *recv_ml = (float2 *)(kv_s + CF::RING + 512);
  float2 *ml = (float2 *)(kv_s + CF::ML_OFF);           // [group][row]
  const int out_f32 = a.out_f32;
  const int r0 = min(kTile, crank * rpc), r1 = min(kTile, r0 + rpc);   // the rows this CTA writes
  const int seg_own = seg_rows(crank);                  // of which the merged ones: [r0, r0 + seg_own)
  constexpr int DHALF = D / 2;                         // a softmax thread's columns [g D/2, (g + 1) D/2)
  float v[DHALF];
  float Mrow = kNegInf, Lrow = 0.f;                    // the CTA's row: max (raw score units), sum
  const int owner = r / rpc;                           // the CTA that writes row r
  const bool merged = C > 1 && owner < C && r - owner * rpc < seg_rows(owner);
  if (warp >= 4) {
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    ml[g * kTile + r] = make_float2(m_run, ok ? l_run : 0.f);
    quadrant_bar(q);
    const float2 ml0 = ml[r], ml1 = ml[kTile + r];
    Mrow = fmaxf(ml0.y > 0.f ? ml0.x : kNegInf, ml1.y > 0.f ? ml1.x : kNegInf);
    const float w0 = ml0.y > 0.f ? tc::ex2_approx((ml0.x - Mrow) * a.scale_log2) : 0.f;
    const float w1 = ml1.y > 0.f ? tc::ex2_approx((ml1.x - Mrow) * a.scale_log2) : 0.f;
    Lrow = w0 * ml0.y + w1 * ml1.y;
    // a quadrant whose rows are all padding (past the rows that can hold a query) reads nothing
    if (q * 32 < pl.nvr) {
#pragma unroll
      for (int c0 = 0; c0 < DHALF; c0 += 32) {
        uint32_t o0[32], o1[32];
        tc::tmem_ld_32x32b_x32(tmem + lane_base + CF::O_COL + (uint32_t)(g * DHALF + c0), o0);
        tc::tmem_ld_32x32b_x32(tmem + lane_base + CF::O_COL + (uint32_t)(D + g * DHALF + c0), o1);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          v[c0 + e] = (w0 > 0.f ? w0 * __uint_as_float(o0[e]) : 0.f) + (w1 > 0.f ? w1 * __uint_as_float(o1[e]) : 0.f);
      }
    } else {
#pragma unroll
      for (int e = 0; e < DHALF; ++e) v[e] = 0.f;
    }
    if (merged && owner != crank) {
      // a merged row another CTA writes: this half row (g) normalised and, from group 0, (max, sum);
      // 16-byte chunk j of row r goes to chunk j ^ (r & 7), so that a warp's 32 rows spread over the banks
      unsigned char *row = send + (size_t)r * CF::RB;
      const float inv = Lrow > 0.f ? 1.f / Lrow : 0.f;
#pragma unroll
      for (int c = 0; c < DHALF / 4; ++c)
        *(float4 *)(row + (((g * DHALF / 4 + c) ^ (r & 7)) * 16)) =
            make_float4(v[4 * c] * inv, v[4 * c + 1] * inv, v[4 * c + 2] * inv, v[4 * c + 3] * inv);
      if (g == 0) send_ml[r] = make_float2(Lrow > 0.f ? Mrow * a.scale_log2 : kNegInf, Lrow);
      tc::fence_proxy_async_smem();                    // the bulk copies read these rows
    }
  }

  if (C > 1) {
    // ---- split merge through the cluster: the merged rows go to their owners ----
    // Each owner receives its rows from every peer into the ring stages the pipeline left out, so no
    // CTA waits for a peer to finish before sending; the cluster barrier begun at the start only
    // ensures that every peer's merge barrier has been initialised.
    tc::cluster_wait();
    // Warp 3 (idle by now) sends: the thread that issues the copies would otherwise be held at its next
    // proxy fence (before the output stores) until they have landed.
    if (warp >= 3) send_bar();                         // the rows to send are complete
    if (threadIdx.x == 96) {
      for (int c = 0; c < C; ++c) {
        const int nr = seg_rows(c);
        if (c == crank || nr == 0) continue;
        const int slot = crank < c ? crank : crank - 1;   // this CTA's slot among owner c's peers
        const uint32_t bar = tc::cluster_map(&br.mrg, (uint32_t)c);
        tc::bulk_copy_to_cluster(tc::cluster_map(recv + (size_t)slot * rpc * CF::RB, (uint32_t)c),
                                 send + (size_t)c * rpc * CF::RB, (uint32_t)(nr * CF::RB), bar);
        tc::bulk_copy_to_cluster(tc::cluster_map(recv_ml + slot * rpc, (uint32_t)c), send_ml + c * rpc,
                                 (uint32_t)(nr * 8), bar);
      }
    }
    if (warp >= 4 && merged && owner == crank) {
      // an owned merged row: combine this CTA's part (registers, relative to Mrow) with the peers'
      // normalised copies; weight of source s: L_s 2^(m_s - M), M = max_s m_s (log2 units)
      // The peers' copies of this CTA's rows.  Every peer sends them, after an abort too, so this wait
      // ignores the abort flag: the CTA must not leave while a copy into it is still on its way.
      if (!tc::mbar_wait(&br.mrg, 0)) fail(br, a.err, 221);
      const float mown = Lrow > 0.f ? Mrow * a.scale_log2 : kNegInf;
      float M = mown;
      for (int sl = 0; sl < C - 1; ++sl) {
        const float2 mlc = recv_ml[sl * rpc + r - r0];
        if (mlc.y > 0.f) M = fmaxf(M, mlc.x);
      }
      const float wown = Lrow > 0.f ? tc::ex2_approx(mown - M) : 0.f;
      float W = wown * Lrow;
#pragma unroll
      for (int e = 0; e < DHALF; ++e) v[e] = wown > 0.f ? v[e] * wown : 0.f;
      for (int sl = 0; sl < C - 1; ++sl) {
        const float2 mlc = recv_ml[sl * rpc + r - r0];
        if (!(mlc.y > 0.f)) continue;                  // an empty split: its values may be anything
        const float wc = mlc.y * tc::ex2_approx(mlc.x - M);
        W += wc;
        const uint32_t rowa = tc::smem_u32(recv + (size_t)(sl * rpc + r - r0) * CF::RB);
#pragma unroll
        for (int cc = 0; cc < DHALF / 4; ++cc) {
          const float4 x = lds_f4(rowa + (uint32_t)(((g * DHALF / 4 + cc) ^ (r & 7)) * 16));
          v[4 * cc] = fmaf(x.x, wc, v[4 * cc]); v[4 * cc + 1] = fmaf(x.y, wc, v[4 * cc + 1]);
          v[4 * cc + 2] = fmaf(x.z, wc, v[4 * cc + 2]); v[4 * cc + 3] = fmaf(x.w, wc, v[4 * cc + 3]);
        }
      }
      // v is now relative to M with sum W (log2 units): as if this CTA had seen every key
      Mrow = M / a.scale_log2;
      Lrow = W;
    }
    // every copy into this CTA has landed (its merging threads waited for them); the barrier completes
    // before any CTA of the cluster leaves, so no copy ever targets a CTA that has exited
    tc::cluster_arrive_relaxed();
  }

  // ---- output: this CTA's rows [r0, r1) ----
  if (warp >= 4 && r >= r0 && r < r1) {
    const float inv = Lrow > 0.f ? 1.f / Lrow : 0.f;
    int hs, qi;
    const bool valid = row_target(pl, a.nq, nh, q0, r, hs, qi);
    const int h = kvh * a.group + h0 + hs;
    if (valid && g == 0 && a.lse && Lrow > 0.f)
      a.lse[((int64_t)b * a.nq + qi) * a.hq + h] = Mrow * a.scale + __logf(Lrow);
    // the normalised half row straight to the output: 16-byte stores, a row's 128 or 256 bytes
    // contiguous (measured faster than staging the tile for TMA stores, at every workload shape)
    if (valid) {
      const int64_t obase = (((int64_t)b * a.nq + qi) * a.hq + h) * D + g * DHALF;
      void *dst = out_f32 ? (void *)((float *)a.out + obase) : (void *)((__nv_bfloat16 *)a.out + obase);
      store_row_part<DHALF>(dst, out_f32 != 0, v, inv);
    }
  }
  // with a cluster, every copy this CTA sent has landed once the exit barrier completes
  if (C > 1) tc::cluster_wait();

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, CF::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// [batch, rows, heads, d] bf16 with the given batch stride (elements), box {64, 1, box_rows, 1}.
bool map4(CUtensorMap *m, const void *base, int d, int heads, int rows, int batch, int64_t batch_stride,
          int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)batch};
  const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2, (cuuint64_t)batch_stride * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K or V [batch, rows, heads, d] viewed as (d, rows, heads, batch) -- rows and heads swapped -- with box
// {64, box_rows, kvp, 1}: one load brings box_rows keys of kvp consecutive heads, head-major, which is
// the tile layout the kernel uses (row p * box_rows + key of head kvh + p).  bf16 with the 128-byte
// swizzle, or E4M3 codes (codes = true: whole d-byte rows, no swizzle: the softmax groups read them by
// half rows).  batch_stride is in elements.
bool map4_kv(CUtensorMap *m, const void *base, int d, int heads, int rows, int batch, int64_t batch_stride,
             int box_rows, int kvp, bool codes) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t es = codes ? 1 : 2;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)heads, (cuuint64_t)batch};
  const cuuint64_t strides[3] = {(cuuint64_t)heads * d * es, (cuuint64_t)d * es, (cuuint64_t)batch_stride * es};
  const cuuint32_t box[4] = {codes ? (cuuint32_t)d : 64u, (cuuint32_t)box_rows, (cuuint32_t)kvp, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, codes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            codes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

Plan make_plan(const AttnProblem &p) {
  Plan pl;
  pl.f0 = p.fresh0;
  pl.f1 = p.fresh0 + p.nq;
  const int group = p.hq / p.hkv;
  // MHA with few queries may pack 2 or 4 KV heads into the 128 rows (each a block of the score tile):
  // no padding rows and fewer CTAs, but 2-4x the key tiles per CTA.  Measured on GB300, it pays only
  // when the unpacked units (one per sequence and KV head) need more than one wave of CTAs; then the
  // smallest packing that fits them in one wave is best (batch 8: 2 heads per tile, 43.6 us instead of
  // 52.6; batch 16: 2 or 4, 60.8 us instead of 75.4; batch 1 or 4: unpacked).
  pl.kvp = 1;
  if (group == 1) {
    const int sms = sm_count();
    for (int kvp = 1; kvp <= 4; kvp *= 2) {
      if (p.nq > kTile / kvp || p.hkv % kvp != 0) break;
      pl.kvp = kvp;
      if (p.batch * (p.hkv / kvp) <= sms) break;
    }
  }
  pl.tk = kKeys / pl.kvp;
  pl.ka = (pl.f0 + pl.tk - 1) / pl.tk;
  pl.kf = (p.nq + pl.tk - 1) / pl.tk;
  pl.kcn = (p.seq_len - pl.f1 + pl.tk - 1) / pl.tk;
  pl.kt = pl.ka + pl.kf + pl.kcn;
  // fewer fresh rows than a tile, and the suffix's last tile short enough to complete theirs: one joined
  // tile (single-head tiles of a bf16 cache, blocks at the same position in every sequence)
  pl.join = 0;
  const int suffix = p.seq_len - pl.f1;
  if (pl.kvp == 1 && !p.f8kv && p.blocks == nullptr && p.nq < pl.tk && p.nq % 8 == 0 && suffix > 0 &&
      suffix % pl.tk > 0 && p.nq + suffix % pl.tk <= pl.tk) {
    pl.join = suffix % pl.tk;
    pl.kcn = suffix / pl.tk;
    pl.kt = pl.ka + pl.kf + pl.kcn;
  }
  if (pl.kvp > 1) {
    pl.qr = kTile / pl.kvp;
    pl.ht = pl.kvp;
    pl.qtiles_per_head = 0;
    pl.nqt = 1;
  } else if (p.nq <= kTile) {
    pl.qr = (p.nq + 7) / 8 * 8;
    pl.ht = kTile / pl.qr;
    pl.qtiles_per_head = 0;
    pl.nqt = (group + pl.ht - 1) / pl.ht;
  } else {
    pl.qr = kTile;
    pl.ht = 1;
    pl.qtiles_per_head = (p.nq + kTile - 1) / kTile;
    pl.nqt = group * pl.qtiles_per_head;
  }
  pl.units = p.batch * (p.hkv / pl.kvp) * pl.nqt;
  pl.abs_suffix = p.blocks != nullptr;
  // per-sequence blocks: a sequence has at most ceil(N / tk) + 2 key tiles (two ragged boundaries)
  const int kt_max = p.blocks != nullptr ? (p.seq_len + pl.tk - 1) / pl.tk + 2 : pl.kt;
  // split the key tiles of a unit over a cluster only as far as it fills idle SMs
  int ns = sm_count() / pl.units;
  if (ns > kMaxCluster) ns = kMaxCluster;
  if (ns > kt_max) ns = kt_max;
  // Split merge: the tile rows that can hold a query (in any unit) are owned by the cluster's CTAs in
  // equal shares of whole 8-row groups.  An owner receives its peers' copies in ring stages taken out
  // of the K/V pipeline (at most kMergeStages) and their (max, sum) pairs after the barriers; a cluster
  // whose copies would not fit is made smaller.
  pl.nvr = pl.kvp > 1 || pl.qtiles_per_head != 0 ? kTile : std::min(pl.ht, group) * pl.qr;
  const int stage = 2 * kKeys * p.d * 2, nstages = p.d == 128 ? Cfg<128>::NS : Cfg<64>::NS;
  auto rows_per = [&](int c) { return ((pl.nvr + c - 1) / c + 7) / 8 * 8; };
  auto merge_stages = [&](int c) {
    const int64_t bytes = (int64_t)(c - 1) * rows_per(c) * p.d * 4;
    return (int)((bytes + stage - 1) / stage);
  };
  while (ns > 1 && (merge_stages(ns) > kMergeStages || (ns - 1) * rows_per(ns) * 8 > Cfg<128>::RECV_ML_BYTES)) --ns;
  pl.nsplit = ns < 1 ? 1 : ns;
  pl.rpc = pl.nsplit > 1 ? rows_per(pl.nsplit) : kTile;
  pl.nsp = nstages - (pl.nsplit > 1 ? merge_stages(pl.nsplit) : 0);
  return pl;
}

// Rows per cache-window store box: whole key tiles of one KV head's keys (tk rows, the block a multiple
// of tk), or the block alone inside one tile of a single head; 0 when neither holds.
int update_box_rows(const Plan &pl, int win) {
  if (win % pl.tk == 0) return pl.tk;
  if (win < pl.tk && pl.kvp == 1) return win;
  return 0;
}

template <int D, int KVP, bool F8KV>
cudaError_t launch_d(const Plan &pl, const CUtensorMap *maps, const Args &a, cudaStream_t st) {
  auto k = attn_tc_kernel<D, KVP, F8KV>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.units * pl.nsplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)pl.nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // prologue overlaps the previous kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, k, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8],
                         maps[9], maps[10], a);
  count_launches(1);
  return e;
}

}  // namespace

template <bool F8KV>
cudaError_t dispatch_kvp(int d, const Plan &pl, const CUtensorMap *maps, const Args &a, cudaStream_t st) {
  if (d == 128) {
    if (pl.kvp == 4) return launch_d<128, 4, F8KV>(pl, maps, a, st);
    if (pl.kvp == 2) return launch_d<128, 2, F8KV>(pl, maps, a, st);
    return launch_d<128, 1, F8KV>(pl, maps, a, st);
  }
  if (pl.kvp == 4) return launch_d<64, 4, F8KV>(pl, maps, a, st);
  if (pl.kvp == 2) return launch_d<64, 2, F8KV>(pl, maps, a, st);
  return launch_d<64, 1, F8KV>(pl, maps, a, st);
}

bool attn_tc_supported(const AttnProblem &p) { return p.in_bf16 && (p.d == 64 || p.d == 128); }

bool attn_tc_fuses_update(const AttnProblem &p) {
  return attn_tc_supported(p) && !p.f8kv && update_box_rows(make_plan(p), p.win) > 0;
}

size_t attn_tc_workspace(const AttnProblem &) { return 0; }

cudaError_t launch_attn_tc(const AttnProblem &p, cudaStream_t st) {
  const Plan pl = make_plan(p);
  const int group = p.hq / p.hkv;
  const int64_t cstride = (int64_t)p.seq_len * p.hkv * p.d;  // cache batch stride
  const int64_t fstride = (int64_t)p.nq * p.hkv * p.d;       // fresh batch stride
  const int64_t qstride = (int64_t)p.nq * p.hq * p.d;
  CUtensorMap maps[11];
  const __nv_bfloat16 *kc = (const __nv_bfloat16 *)p.kc, *vc = (const __nv_bfloat16 *)p.vc;
  // per-sequence blocks: prefix and suffix tiles are read through maps of the whole cache; rows of a
  // sequence's own window that fall in a boundary tile are read and weighted by exactly zero
  const bool per_seq = p.blocks != nullptr;
  const int64_t off_c = per_seq ? 0 : (int64_t)pl.f1 * p.hkv * p.d;
  const int rows_a = per_seq ? p.seq_len : pl.f0, rows_c = per_seq ? p.seq_len : p.seq_len - pl.f1;
  const int kvp = pl.kvp;
  // a joined tile reads the fresh rows as one box of nq rows
  const int fbox = pl.join > 0 ? p.nq : pl.tk;
  bool ok = map4(&maps[0], p.q, p.d, p.hq, p.nq, p.batch, qstride, pl.qr) &&
            map4_kv(&maps[2], p.kf, p.d, p.hkv, p.nq, p.batch, fstride, fbox, kvp, false) &&
            map4_kv(&maps[5], p.vf, p.d, p.hkv, p.nq, p.batch, fstride, fbox, kvp, false);
  if (p.f8kv) {   // the cache as E4M3 codes (one byte per element)
    const uint8_t *kq = (const uint8_t *)p.kc, *vq = (const uint8_t *)p.vc;
    ok = ok && map4_kv(&maps[1], kq, p.d, p.hkv, rows_a, p.batch, cstride, pl.tk, kvp, true) &&
         map4_kv(&maps[3], kq + off_c, p.d, p.hkv, rows_c, p.batch, cstride, pl.tk, kvp, true) &&
         map4_kv(&maps[4], vq, p.d, p.hkv, rows_a, p.batch, cstride, pl.tk, kvp, true) &&
         map4_kv(&maps[6], vq + off_c, p.d, p.hkv, rows_c, p.batch, cstride, pl.tk, kvp, true);
  } else {
    ok = ok && map4_kv(&maps[1], p.kc, p.d, p.hkv, rows_a, p.batch, cstride, pl.tk, kvp, false) &&
         map4_kv(&maps[3], kc + off_c, p.d, p.hkv, rows_c, p.batch, cstride, pl.tk, kvp, false) &&
         map4_kv(&maps[4], p.vc, p.d, p.hkv, rows_a, p.batch, cstride, pl.tk, kvp, false) &&
         map4_kv(&maps[6], vc + off_c, p.d, p.hkv, rows_c, p.batch, cstride, pl.tk, kvp, false);
  }
  // the cache-window store maps: the whole caches, boxes of win_box rows (unused copies otherwise)
  int win_box = 0;
  if (p.update) {
    win_box = update_box_rows(pl, p.win);
    if (win_box > 0)
      ok = ok && map4_kv(&maps[7], p.kc_w, p.d, p.hkv, p.seq_len, p.batch, cstride, win_box, kvp, false) &&
           map4_kv(&maps[8], p.vc_w, p.d, p.hkv, p.seq_len, p.batch, cstride, win_box, kvp, false);
  }
  if (win_box == 0) maps[7] = maps[8] = maps[1];
  // the joined tile's suffix rows: the suffix maps with boxes of tk - nq rows (unused copies otherwise)
  if (pl.join > 0)
    ok = ok && map4_kv(&maps[9], kc + off_c, p.d, p.hkv, rows_c, p.batch, cstride, pl.tk - p.nq, kvp, false) &&
         map4_kv(&maps[10], vc + off_c, p.d, p.hkv, rows_c, p.batch, cstride, pl.tk - p.nq, kvp, false);
  else
    maps[9] = maps[10] = maps[3];
  if (!ok) return cudaErrorInvalidValue;
  Args a;
  a.win = p.update ? p.win : 0;
  a.win_box = win_box;
  a.pl = pl;
  a.batch = p.batch; a.n = p.seq_len; a.nq = p.nq; a.hq = p.hq; a.hkv = p.hkv; a.group = group;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  a.out_f32 = p.out_f32;
  a.out = p.out;
  a.lse = p.lse;
  a.err = p.err;
  a.blocks = p.blocks;
  a.prompt_len = p.prompt_len;
  a.nblocks = p.nblocks;
  a.k_scale = p.k_scale;
  a.v_scale = p.v_scale;
  if (p.f8kv) return dispatch_kvp<true>(p.d, pl, maps, a, st);
  return dispatch_kvp<false>(p.d, pl, maps, a, st);
}

}  // namespace fdllm
