// Block attention on the 5th-generation tensor cores (bf16 in, fp32 accumulate).
//
// Keys are taken as three contiguous ranges, each through its own TMA map so
// that no row outside a range is ever read: the cached prefix [0, f0), the fresh
// keys of this step (nq rows, the query positions) and the cached suffix
// [f1, N).  Softmax is invariant to the order of the keys, so the key tiles of
// 64 rows are enumerated range by range.
//
// One CTA = (sequence, KV head, 128-row query tile, split of the key tiles);
// all query heads sharing the KV head are packed into the 128 rows when
// nq <= 128.  Within the CTA the key tiles are pipelined:
//   warp 0     TMA: the query tile once, then K and V tiles into a ring
//   warp 1     TMEM owner, MMA issuer: S_i = Q K_i^T (M=128, N=64 keys,
//              K=d) into one of two TMEM score buffers, then PV_i = P_i V_i
//              (N=d, K=64 keys, V read MN-major) into one of two TMEM
//              buffers; S_{i+1} is issued before PV_i; the K/V ring holds
//              4 tiles (d = 128) so loads run ahead of the MMAs
//   warps 4-11 two threads per query row (warps w and w + 4 share a TMEM lane
//              quadrant and split the key and output columns; they exchange
//              the half-row maxima through shared memory under a barrier of
//              the two warps only), online softmax in base 2 with a lazy
//              reference max: P_i = 2^(S_i - m_ref) is written as bf16 (128-byte
//              swizzle) into one of two P buffers and the tensor core
//              accumulates O += P_i V_i in TMEM.  m_ref moves only when a row's
//              max exceeds it by more than 2^8; then that row of O (and l) is
//              rescaled in TMEM once the previous PV product has landed.
//              Tile i+1's softmax runs while the tensor core computes PV_i.
// Splits of one unit form a thread block cluster (<= 8) and merge through
// distributed shared memory with stores only, between two cluster barriers:
// every CTA writes each of its O rows, unnormalised, with the row's (max, l)
// into the CTA that owns the row (CTA c owns rows [c R/C, (c+1) R/C)), and each
// owner combines the C copies of its rows with weights 2^(m_c - M) / L and
// writes them.
//
// K/V maps view [b, N, Hkv, d] as (d, position, head, b), so one box brings a
// tile half's keys of all heads packed in the tile, head-major.
//
// FP8 KV cache (F8KV): cached K and V are E4M3 codes with one power-of-two scale
// per (sequence, position, KV head) row.  A cache tile is loaded as bytes into
// the V half of its ring stage; warps 2-3 (one thread per key row) turn the K
// codes into the bf16 K tile TMA would have written -- code * scale is exact in
// bf16 -- and release it to the MMA issuer; the softmax warps turn the V codes
// into the bf16 V tile at the start of the tile's softmax.  The products and the
// softmax arithmetic are unchanged.  Fresh K/V tiles are loaded as bf16 directly.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 384;   // warps 0-3: TMA, MMA, FP8 K conversion (2, 3); 4-11: softmax (two per quadrant)
constexpr int kTile = 128;       // rows per query tile
constexpr int kKeys = 64;        // keys per key tile
constexpr int kMaxCluster = 8;   // portable thread-block cluster size
constexpr float kLog2e = 1.4426950408889634f;

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
};

template <int D>
struct Cfg {
  static constexpr int DH = D / 64;                   // 64-column halves of a row
  static constexpr int Q_BYTES = kTile * D * 2;       // 128 query rows x d bf16
  static constexpr int QHALF = kTile * 128;           // 128 rows x 64 bf16
  static constexpr int KV_BYTES = kKeys * D * 2;      // 64 key rows x d bf16
  static constexpr int KVHALF = kKeys * 128;          // 64 rows x 64 bf16
  static constexpr int P_BYTES = kTile * kKeys * 2;   // 128 rows x 64 keys bf16 (one swizzle atom column)
  static constexpr int STAGE = 2 * KV_BYTES;          // K + V
  static constexpr int NS = D == 128 ? 4 : 8;         // K/V ring stages
  // cluster merge: the O rows an owner receives, C * ceil(128 / C) <= 136 of them, fp32 with a row
  // pitch of D + 4 floats (a column written by 8 consecutive rows falls in 8 different banks), then
  // each received row's (max, l), then its combination weight
  static constexpr int MERGE_ROWS = 136;
  static constexpr int DP = D + 4;
  static constexpr int MERGE_BYTES = MERGE_ROWS * DP * 4 + MERGE_ROWS * 8 + MERGE_ROWS * 4;
  static constexpr int RING = NS * STAGE > MERGE_BYTES ? NS * STAGE : MERGE_BYTES;
  static constexpr int SMEM = Q_BYTES + RING + 2 * P_BYTES + 1024 + 4096;   // + alignment + Bars
  static constexpr uint32_t S_COL = 0;                // TMEM: S0, S1 (64 columns each), then O (D columns)
  static constexpr uint32_t O_COL = 2 * kKeys;
  static constexpr uint32_t TMEM_COLS = 256;
};

struct Bars {
  uint64_t qfull, kvfull[8], kvempty[8], sfull[2], sempty[2], pfull[2], pvdone, drain;
  uint64_t raw[8];     // F8KV: a cache tile's codes have landed (the converters then complete kvfull)
  uint32_t tmem_base;
  int32_t cvt_stop;   // F8KV: the converters stop (written before, read between their two barriers)  // (the whole struct must fit the 4096 bytes reserved after the P buffers)
  int32_t abort;
  int32_t issued;     // K/V tiles issued by the producer
  int32_t consumed;   // K/V tiles whose arrival the MMA issuer waited for
  float rowmax[2][2][kTile];  // [tile parity][column half][row] half-row maxima
  float lhalf[2][kTile];      // [column half][row] partial softmax denominators
};

// The 256 softmax threads (warps 4-11) synchronise among themselves.
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The two softmax warps of TMEM lane quadrant q (warps 4 + q and 8 + q) synchronise as a pair.
__device__ __forceinline__ void quadrant_bar(int q) { asm volatile("bar.sync %0, 64;" ::"r"(2 + q) : "memory"); }

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
    t.range = 1; t.row0 = (k - pl.ka) * pl.tk; t.nvalid = min(pl.tk, nq - t.row0);
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
};

// The two FP8 conversion warps synchronise among themselves.
__device__ __forceinline__ void convert_bar() { asm volatile("bar.sync 6, 64;" ::: "memory"); }

// 4 E4M3 codes (one 32-bit word) times `sc` as 4 bf16 (two words); exact: an E4M3 value has at most
// 4 significant bits and `sc` is a power of two.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w, float sc) {
  uint32_t o[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> (16 * h)), __NV_E4M3);
    const float2 f = __half22float2(*(const __half2 *)&hr);
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc, f.y * sc);
    o[h] = *(const uint32_t *)&b;
  }
  return make_uint2(o[0], o[1]);
}

// Row r of a bf16 K or V tile in the layout the 128-byte-swizzled TMA load writes: 64-column halves
// of kKeys rows x 128 bytes, 16-byte chunk j of row r at chunk j ^ (r & 7).  `codes` holds the row's
// D / 16 chunks of 16 codes; chunk slot c holds code chunk (c + r) mod (D / 16) (the rotation
// spreads a warp's shared-memory accesses over the banks).
template <int D>
__device__ __forceinline__ void store_bf16_row(unsigned char *tile, int r, const uint4 (&codes)[D / 16], float sc) {
  constexpr int NC = D / 16;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int cc = (c + r) & (NC - 1);
    const uint2 a = e4m3x4_to_bf16x4(codes[c].x, sc), b = e4m3x4_to_bf16x4(codes[c].y, sc);
    const uint2 d = e4m3x4_to_bf16x4(codes[c].z, sc), e = e4m3x4_to_bf16x4(codes[c].w, sc);
    unsigned char *half = tile + (cc >> 2) * (kKeys * 128) + r * 128;
    const int j = (cc & 3) * 2;                      // first of the two 16-byte bf16 chunks
    *(uint4 *)(half + ((j ^ (r & 7)) * 16)) = make_uint4(a.x, a.y, b.x, b.y);
    *(uint4 *)(half + (((j + 1) ^ (r & 7)) * 16)) = make_uint4(d.x, d.y, e.x, e.y);
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

template <int D>
__device__ __forceinline__ void load_code_row(const unsigned char *row, int r, uint4 (&codes)[D / 16]) {
  constexpr int NC = D / 16;
#pragma unroll
  for (int c = 0; c < NC; ++c) codes[c] = *(const uint4 *)(row + ((c + r) & (NC - 1)) * 16);
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

static_assert(sizeof(Bars) <= 4096, "Bars must fit its shared-memory reservation");

template <int D, int KVP, bool F8KV>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mka,
                   const __grid_constant__ CUtensorMap mkf, const __grid_constant__ CUtensorMap mkc,
                   const __grid_constant__ CUtensorMap mva, const __grid_constant__ CUtensorMap mvf,
                   const __grid_constant__ CUtensorMap mvc, const Args a) {
  using CF = Cfg<D>;
  constexpr int NS = CF::NS;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *q_s = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char *kv_s = q_s + CF::Q_BYTES;              // NS stages of (K tile, V tile)
  unsigned char *p_s = kv_s + CF::RING;                 // 2 P buffers
  Bars &br = *(Bars *)(p_s + 2 * CF::P_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Plan pl = a.pl;   // per-sequence blocks fill in this CTA's ranges after the dependency wait

  const int split = blockIdx.x % pl.nsplit;
  const int unit = blockIdx.x / pl.nsplit;
  const int nkvg = a.hkv / KVP;                        // KV head groups
  const int qt = unit % pl.nqt;
  const int kvh = ((unit / pl.nqt) % nkvg) * KVP;        // first KV head of this tile
  const int b = unit / (pl.nqt * nkvg);
  int h0, nh, q0;
  if (KVP > 1) {
    h0 = 0; nh = KVP; q0 = 0;                          // head slot s = KV head kvh + s (MHA)
  } else if (pl.qtiles_per_head == 0) {
    h0 = qt * pl.ht; nh = min(pl.ht, a.group - h0); q0 = 0;
  } else {
    h0 = qt / pl.qtiles_per_head; nh = 1; q0 = (qt % pl.qtiles_per_head) * kTile;
  }

  if (threadIdx.x == 0) {
    br.abort = 0; br.issued = 0; br.consumed = 0; br.cvt_stop = 0;
    tc::mbar_init(&br.qfull, 1);
    for (int i = 0; i < NS; ++i) { tc::mbar_init(&br.kvfull[i], 1); tc::mbar_init(&br.kvempty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&br.sfull[i], 1);
      tc::mbar_init(&br.sempty[i], 8);
      tc::mbar_init(&br.pfull[i], 8);
    }
    tc::mbar_init(&br.pvdone, 1);
    tc::mbar_init(&br.drain, 1);
    for (int i = 0; i < NS; ++i) tc::mbar_init(&br.raw[i], 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&br.tmem_base, CF::TMEM_COLS);
  if (threadIdx.x == 0) {
    for (const CUtensorMap *m : {&mq, &mka, &mkf, &mkc, &mva, &mvf, &mvc}) tc::prefetch_tensormap(m);
  }
  if (KVP > 1) {
    // each row writes only its own head's block of a P tile: the rest stays zero
    for (int i = threadIdx.x; i < 2 * CF::P_BYTES / 16; i += kThreads) ((uint4 *)p_s)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc::fence_proxy_async_smem();
  }
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

  // thread of the softmax warps: its query row, column half and running state (reference max, l)
  const int r = (warp & 3) * 32 + lane;
  const int half = (warp - 4) >> 2;
  float m_run = kNegInf, l_run = 0.f;
  // set by the first wait that gives up (fail()); every later wait that polls it returns at once
  const volatile int32_t *abort_flag = &br.abort;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_q = tc::policy_evict_last();
      const uint64_t pol_kv = tc::policy_evict_first();
      tc::mbar_arrive_expect_tx(&br.qfull, (uint32_t)(pl.qr * 128 * CF::DH * nh));
      for (int hs = 0; hs < nh; ++hs)
        for (int dh = 0; dh < CF::DH; ++dh)
          tc::tma_load_4d(q_s + dh * CF::QHALF + hs * pl.qr * 128, &mq, &br.qfull, dh * 64,
                          kvh * a.group + h0 + hs, q0, b, pol_q);
      for (int i = 0; i < nt && !br.abort; ++i) {
        const int st = i % NS;
        if (!tc::mbar_wait_or_abort(&br.kvempty[st], ((uint32_t)(i / NS) & 1u) ^ 1u, abort_flag)) {
          if (!*abort_flag) fail(br, a.err, 211);
          break;
        }
        const KeyTile kt = key_tile(pl, a.nq, a.n, k0 + i);
        const CUtensorMap *mk = kt.range == 0 ? &mka : (kt.range == 1 ? &mkf : &mkc);
        const CUtensorMap *mv = kt.range == 0 ? &mva : (kt.range == 1 ? &mvf : &mvc);
        unsigned char *ks = kv_s + st * CF::STAGE;
        if (F8KV && kt.range != 1) {
          // cache tile: K codes then V codes (kKeys rows x D bytes each) into the stage's V half; the
          // converters write the bf16 tiles and complete kvfull
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
          }
        }
        atomicExch(&br.issued, i + 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_bf16_f32(128, kKeys, 0);
      const uint32_t id_o = tc::idesc_bf16_f32(128, D, 1);
      const uint32_t qa = tc::smem_u32(q_s);
      bool ok = tc::mbar_wait_or_abort(&br.qfull, 0, abort_flag);
      if (!ok && !*abort_flag) fail(br, a.err, 212);
      auto issue_s = [&](int i) -> bool {
        const int st = i % NS, j = i & 1;
        if (!tc::mbar_wait_or_abort(&br.kvfull[st], (uint32_t)(i / NS) & 1u, abort_flag)) {
          if (!*abort_flag) fail(br, a.err, 213);
          return false;
        }
        atomicExch(&br.consumed, i + 1);
        if (!tc::mbar_wait_or_abort(&br.sempty[j], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag)) {
          if (!*abort_flag) fail(br, a.err, 214);
          return false;
        }
        tc::fence_after_sync();
        const uint32_t ka = tc::smem_u32(kv_s + st * CF::STAGE);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t kin = (uint32_t)((ks % 4) * 32);
          tc::mma_bf16(tmem + CF::S_COL + (uint32_t)(j * kKeys), tc::sw128_desc(qa + (ks / 4) * CF::QHALF + kin),
                       tc::sw128_desc(ka + (ks / 4) * CF::KVHALF + kin), id_s, ks != 0);
        }
        tc::mma_commit(&br.sfull[j]);
        return true;
      };
      auto issue_pv = [&](int i) -> bool {
        const int st = i % NS, j = i & 1;
        if (!tc::mbar_wait_or_abort(&br.pfull[j], (uint32_t)(i >> 1) & 1u, abort_flag)) {
          if (!*abort_flag) fail(br, a.err, 215);
          return false;
        }
        tc::fence_after_sync();
        const uint32_t pa = tc::smem_u32(p_s + j * CF::P_BYTES);
        const uint32_t va = tc::smem_u32(kv_s + st * CF::STAGE + CF::KV_BYTES);
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks)
          tc::mma_bf16(tmem + CF::O_COL, tc::sw128_desc(pa + (uint32_t)(ks * 32)),
                       tc::sw128_mn_desc(va + (uint32_t)(ks * 2048), CF::KVHALF), id_o, (i | ks) != 0);
        tc::mma_commit(&br.pvdone);
        tc::mma_commit(&br.kvempty[st]);
        return true;
      };
      if (ok && nt > 0) ok = issue_s(0);
      for (int i = 0; i < nt && ok; ++i) {
        if (i + 1 < nt && !issue_s(i + 1)) break;
        if (!issue_pv(i)) break;
      }
      tc::mma_commit(&br.drain);
      if (!tc::mbar_wait(&br.drain, 0)) record_device_error(a.err, 217);
    }
  } else if (F8KV && (warp == 2 || warp == 3)) {
    // FP8 cache K tiles to bf16: thread r converts key row r (KV head kvh + r / tk, key r % tk)
    const int r = threadIdx.x - 64;
    // Every converter thread takes each exit decision from cvt_stop, which is only written before the
    // first barrier of an iteration and read between its two barriers: no thread can leave while
    // another waits at a barrier.
    uint32_t rawpar = 0;                               // bit st: parity of raw[st]'s next phase
    // this row's K scale, loaded one cache tile ahead so that its latency overlaps a conversion
    auto next_cache_tile = [&](int j) {
      while (j < nt && key_tile(pl, a.nq, a.n, k0 + j).range == 1) ++j;
      return j;
    };
    auto load_scale = [&](int j) -> float {
      return j < nt ? cache_scale(a, pl, key_tile(pl, a.nq, a.n, k0 + j), b, kvh, r, a.k_scale) : 0.f;
    };
    int inext = next_cache_tile(0);
    float ksn = load_scale(inext);
    for (int i = inext; i < nt; i = inext) {
      const float ksc = ksn;
      inext = next_cache_tile(i + 1);
      ksn = load_scale(inext);
      const int st = i % NS;
      if (!tc::mbar_wait_or_abort(&br.raw[st], (rawpar >> st) & 1u, abort_flag)) {
        if (!*abort_flag) fail(br, a.err, 220);
        br.cvt_stop = 1;
      }
      rawpar ^= 1u << st;
      if (r == 0 && br.abort) br.cvt_stop = 1;
      convert_bar();
      if (br.cvt_stop) break;
      unsigned char *ks = kv_s + st * CF::STAGE;
      uint4 codes[D / 16];
      load_code_row<D>(ks + CF::KV_BYTES + r * D, r, codes);
      store_bf16_row<D>(ks, r, codes, ksc);            // K: codes in the V half, bf16 into the K half
      tc::fence_proxy_async_smem();
      convert_bar();
      if (r == 0) tc::mbar_arrive(&br.kvfull[st]);     // V is converted by the softmax warps
    }
  } else if (warp >= 4) {
    constexpr int DHALF = D / 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t oa = tmem + lane_base + CF::O_COL + (uint32_t)(half * DHALF);   // this thread's O columns
    // Every softmax warp runs every tile and meets every named barrier (the pair's quadrant barrier,
    // the 256-thread softmax barrier) the same number of times, whatever its waits return: a wait that
    // gives up only marks this thread's result invalid (ok = false), records the site and raises the
    // abort flag, after which every wait of the CTA returns at once.  So no warp can be left waiting
    // at a named barrier for a partner that has left the loop.
    bool ok = true;
    // wait until PV_i has been accumulated into O (phases complete in order, one per tile)
    auto wait_pv = [&](int i) {
      if (!tc::mbar_wait_or_abort(&br.pvdone, (uint32_t)i & 1u, abort_flag)) {
        if (!*abort_flag) fail(br, a.err, 219);
        ok = false;
      }
      tc::fence_after_sync();
    };
    // softmax of tile i over this thread's 32 key columns: P_i = 2^((S_i - m_ref) * scale * log2 e)
    uint32_t vrawpar = 0;                            // F8KV: bit st, parity of raw[st]'s next phase
    auto softmax = [&](int i) {
      const int j = i & 1;
      // F8KV: the 256 softmax threads also turn a cache tile's V codes into bf16 (thread t: a quarter of
      // key row t / 4).  S_i is done, so the converters have read this tile's K codes, which the bf16 V
      // rows overwrite; P_i's release (below) covers these writes too.
      const bool cvt_v = F8KV && key_tile(pl, a.nq, a.n, k0 + i).range != 1;
      const int vt = threadIdx.x - 128, vr = vt >> 2, vq = vt & 3;
      float vsc = 0.f;
      if (F8KV && cvt_v) vsc = cache_scale(a, pl, key_tile(pl, a.nq, a.n, k0 + i), b, kvh, vr, a.v_scale);
      if (!tc::mbar_wait_or_abort(&br.sfull[j], (uint32_t)(i >> 1) & 1u, abort_flag)) {
        if (!*abort_flag) fail(br, a.err, 218);
        ok = false;
      }
      tc::fence_after_sync();
      if constexpr (F8KV) {
        if (cvt_v) {
          constexpr int QC = D / 64;                   // 16-code chunks per quarter row
          const int st = i % NS;
          // the codes' arrival, for this thread: complete long ago (the converters waited for it), and
          // raw[st] cannot move on before this tile's P is released
          if (!tc::mbar_wait_or_abort(&br.raw[st], (vrawpar >> st) & 1u, abort_flag)) ok = false;
          vrawpar ^= 1u << st;
          unsigned char *vh = kv_s + st * CF::STAGE + CF::KV_BYTES;
          uint4 cq[QC];
#pragma unroll
          for (int c = 0; c < QC; ++c) cq[c] = *(const uint4 *)(vh + kKeys * D + vr * D + (vq * QC + c) * 16);
          softmax_bar();                               // every V code of the tile has been read
#pragma unroll
          for (int c = 0; c < QC; ++c) {
            const int cc = vq * QC + c;
            const uint2 x0 = e4m3x4_to_bf16x4(cq[c].x, vsc), x1 = e4m3x4_to_bf16x4(cq[c].y, vsc);
            const uint2 x2 = e4m3x4_to_bf16x4(cq[c].z, vsc), x3 = e4m3x4_to_bf16x4(cq[c].w, vsc);
            unsigned char *row = vh + (cc >> 2) * (kKeys * 128) + vr * 128;
            const int jj = (cc & 3) * 2;
            *(uint4 *)(row + ((jj ^ (vr & 7)) * 16)) = make_uint4(x0.x, x0.y, x1.x, x1.y);
            *(uint4 *)(row + (((jj + 1) ^ (vr & 7)) * 16)) = make_uint4(x2.x, x2.y, x3.x, x3.y);
          }
        }
      }
      // this thread's CW score columns: half `half` of its row's head block (the whole tile when
      // KVP == 1; with KVP heads packed, row r's head owns columns [s TK, s TK + TK), s = r / qr)
      constexpr int TK = kKeys / KVP, CW = TK / 2;
      const int c0 = (KVP > 1 ? r / pl.qr : 0) * TK + half * CW;
      const int nv = key_tile(pl, a.nq, a.n, k0 + i).nvalid - half * CW;   // valid columns of this thread
      uint32_t x[CW];
      const uint32_t sa = tmem + lane_base + CF::S_COL + (uint32_t)(j * kKeys + c0);
      if constexpr (CW == 32) tc::tmem_ld_32x32b_x32(sa, x);
      else if constexpr (CW == 16) tc::tmem_ld_32x32b_x16(sa, x);
      else tc::tmem_ld_32x32b_x8(sa, x);
      tc::tmem_ld_wait();
      float mx[CW / 2];                              // half-row max as a tree
#pragma unroll
      for (int e = 0; e < CW / 2; ++e)
        mx[e] = fmaxf(e < nv ? __uint_as_float(x[e]) : kNegInf,
                      e + CW / 2 < nv ? __uint_as_float(x[e + CW / 2]) : kNegInf);
#pragma unroll
      for (int w = CW / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
      br.rowmax[j][half][r] = mx[0];
      quadrant_bar(warp & 3);                        // the other half of these 32 rows
      float tm = fmaxf(br.rowmax[j][0][r], br.rowmax[j][1][r]);
      // move the reference max only when the row max outgrows it by more than 2^8
      const bool need = m_run == kNegInf || (tm - m_run) * a.scale_log2 > 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? fmaxf(m_run, tm) : m_run;
        const float al = tc::ex2_approx((m_run - m_new) * a.scale_log2);   // 0 on a row's first tile
        if (i > 0) {
          wait_pv(i - 1);                          // O holds PV_0 .. PV_{i-1}
#pragma unroll
          for (int c0 = 0; c0 < DHALF; c0 += 32) {
            uint32_t o[32];
            tc::tmem_ld_32x32b_x32(oa + (uint32_t)c0, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * al);
            tc::tmem_st_32x32b_x32(oa + (uint32_t)c0, o);
          }
          tc::tmem_st_wait();
        }
        l_run *= al;
        m_run = m_new;
      }
      const float ms = m_run * a.scale_log2;
      // CW keys = chunks c0 / 8 .. c0 / 8 + CW / 8 - 1 of this row's 128 bytes in the 128-byte swizzle
      // layout (with KVP heads packed, the row's other chunks hold zeros from the prologue)
      unsigned char *rowp = p_s + j * CF::P_BYTES + r * 128;
      float lt[4] = {0.f, 0.f, 0.f, 0.f};           // four independent partial sums
#pragma unroll
      for (int cc = 0; cc < CW / 8; ++cc) {
        const int ch = c0 / 8 + cc;
        uint32_t pk[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int e = cc * 8 + e2 * 2;
          const float p0 = (e < nv) ? tc::ex2_approx(fmaf(__uint_as_float(x[e]), a.scale_log2, -ms)) : 0.f;
          const float p1 = (e + 1 < nv) ? tc::ex2_approx(fmaf(__uint_as_float(x[e + 1]), a.scale_log2, -ms)) : 0.f;
          lt[cc & 3] += p0 + p1;
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pk[e2] = *(uint32_t *)&h2;
        }
        *(uint4 *)(rowp + ((ch ^ (r & 7)) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l_run += (lt[0] + lt[1]) + (lt[2] + lt[3]);
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&br.pfull[j]);
        tc::mbar_arrive(&br.sempty[j]);
      }
    };
    for (int i = 0; i < nt; ++i) softmax(i);
    if (nt > 0) wait_pv(nt - 1);                   // O is complete
    if (!ok) l_run = 0.f;
    br.lhalf[half][r] = l_run;
    softmax_bar();
    l_run = ok ? br.lhalf[0][r] + br.lhalf[1][r] : 0.f;
    if (pl.nsplit == 1 && ok && l_run > 0.f) {
      int hs, qi;
      const bool valid = row_target(pl, a.nq, nh, q0, r, hs, qi);
      const int h = kvh * a.group + h0 + hs;
      const float inv = 1.f / l_run;
      const int64_t obase = (((int64_t)b * a.nq + qi) * a.hq + h) * D + half * DHALF;
#pragma unroll
      for (int c0 = 0; c0 < DHALF; c0 += 32) {
        uint32_t x[32];
        tc::tmem_ld_32x32b_x32(oa + (uint32_t)c0, x);
        tc::tmem_ld_wait();
        if (!valid) continue;
        if (a.out_f32) {
          float4 *dst = (float4 *)((float *)a.out + obase + c0);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(x[4 * q4]) * inv, __uint_as_float(x[4 * q4 + 1]) * inv,
                                  __uint_as_float(x[4 * q4 + 2]) * inv, __uint_as_float(x[4 * q4 + 3]) * inv);
        } else {
          uint4 *dst = (uint4 *)((__nv_bfloat16 *)a.out + obase + c0);
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(x[8 * q8 + 2 * e]) * inv,
                                                        __uint_as_float(x[8 * q8 + 2 * e + 1]) * inv);
              w[e] = *(uint32_t *)&h2;
            }
            dst[q8] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (valid && half == 0 && a.lse) a.lse[((int64_t)b * a.nq + qi) * a.hq + h] = m_run * a.scale + __logf(l_run);
    }
  }

  if (pl.nsplit > 1) {
    // ---- merge the splits of this unit through the cluster's shared memory, stores only ----
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = pl.nsplit;
    const int crank = (int)cluster.block_rank();
    constexpr int CH = D / 4;                        // float4 chunks per row
    constexpr int DP = CF::DP;
    const int rpc = (kTile + C - 1) / C;             // rows owned per CTA
    // receive area in the K/V ring: [C][rpc] O rows (unnormalised), then [C][rpc] (max * log2 e, l)
    float *orecv = (float *)kv_s;
    float2 *mlrecv = (float2 *)(kv_s + (size_t)CF::MERGE_ROWS * DP * 4);
    tc::fence_before_sync();
    cluster.sync();                                  // every CTA's MMAs and copies are done: rings are free
    if (warp >= 4) {
      // this thread's half row, as accumulated, and the row's (max, l) go to the CTA that owns the row
      const int owner = r / rpc;
      const int slot = crank * rpc + (r - owner * rpc);
      float *orow = orecv + (size_t)slot * DP + half * (D / 2);
      float4 *dst = (float4 *)(owner == crank ? orow : cluster.map_shared_rank(orow, owner));
      if (half == 0) {
        const float2 mine = l_run > 0.f ? make_float2(m_run * a.scale_log2, l_run) : make_float2(kNegInf, 0.f);
        *(owner == crank ? mlrecv + slot : cluster.map_shared_rank(mlrecv + slot, owner)) = mine;
      }
      const uint32_t oa = tmem + ((uint32_t)((warp & 3) * 32) << 16) + CF::O_COL + (uint32_t)(half * (D / 2));
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t x[32];
        tc::tmem_ld_32x32b_x32(oa + (uint32_t)c0, x);
        tc::tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          dst[c0 / 4 + q4] = make_float4(__uint_as_float(x[4 * q4]), __uint_as_float(x[4 * q4 + 1]),
                                         __uint_as_float(x[4 * q4 + 2]), __uint_as_float(x[4 * q4 + 3]));
      }
    }
    cluster.sync();                                  // every row is in its owner
    // owner: out = sum_c O_c w_c with w_c = 2^(m_c - M) / L, M = max_c m_c, L = sum_c l_c 2^(m_c - M)
    const int r0 = crank * rpc, r1 = min(kTile, r0 + rpc);
    float *wrecv = (float *)(mlrecv + CF::MERGE_ROWS);   // [C][rpc] weights, 0 for an empty or aborted split
    for (int lr = threadIdx.x; lr < r1 - r0; lr += kThreads) {
      float M = kNegInf, L = 0.f;
      for (int c = 0; c < C; ++c) M = fmaxf(M, mlrecv[c * rpc + lr].x);
      for (int c = 0; c < C; ++c) {
        const float2 ml = mlrecv[c * rpc + lr];
        if (ml.y > 0.f) L += ml.y * exp2f(ml.x - M);
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int c = 0; c < C; ++c) {
        const float2 ml = mlrecv[c * rpc + lr];
        wrecv[c * rpc + lr] = ml.y > 0.f ? exp2f(ml.x - M) * inv : 0.f;
      }
      int hs, qi;
      if (a.lse && L > 0.f && row_target(pl, a.nq, nh, q0, r0 + lr, hs, qi))
        a.lse[((int64_t)b * a.nq + qi) * a.hq + kvh * a.group + h0 + hs] = (M + log2f(L)) * 0.6931471805599453f;
    }
    __syncthreads();
    for (int u = threadIdx.x; u < (r1 - r0) * CH; u += kThreads) {
      const int lr = u / CH, ch = u % CH;
      int hs, qi;
      if (!row_target(pl, a.nq, nh, q0, r0 + lr, hs, qi)) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = 0; c < C; ++c) {
        const float w = wrecv[c * rpc + lr];
        if (w == 0.f) continue;                      // its rows may hold anything
        const float4 v = *(const float4 *)(orecv + (size_t)(c * rpc + lr) * DP + ch * 4);
        acc.x = fmaf(v.x, w, acc.x); acc.y = fmaf(v.y, w, acc.y);
        acc.z = fmaf(v.z, w, acc.z); acc.w = fmaf(v.w, w, acc.w);
      }
      const int64_t off = (((int64_t)b * a.nq + qi) * a.hq + kvh * a.group + h0 + hs) * D + ch * 4;
      if (a.out_f32) {
        *(float4 *)((float *)a.out + off) = acc;
      } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        *(uint2 *)((__nv_bfloat16 *)a.out + off) = make_uint2(*(uint32_t *)&lo, *(uint32_t *)&hi);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (br.abort && threadIdx.x == 0) {
    // copies issued but never consumed still land in shared memory: wait for them (bounded)
    for (int i = br.consumed; i < br.issued; ++i) {
      if (F8KV && key_tile(pl, a.nq, a.n, k0 + i).range != 1) {
        int uses = 0;                                  // earlier cache tiles in this stage: raw's phase
        for (int j = i % NS; j < i; j += NS) uses += key_tile(pl, a.nq, a.n, k0 + j).range != 1;
        tc::mbar_wait(&br.raw[i % NS], (uint32_t)uses & 1u);
      } else {
        tc::mbar_wait(&br.kvfull[i % NS], (uint32_t)(i / NS) & 1u);
      }
    }
  }
  __syncthreads();
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
// swizzle, or E4M3 codes (codes = true: whole d-byte rows, no swizzle: the converters read them row by
// row).  batch_stride is in elements.
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
  pl.nsplit = ns < 1 ? 1 : ns;
  return pl;
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
  e = cudaLaunchKernelEx(&cfg, k, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], a);
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

size_t attn_tc_workspace(const AttnProblem &) { return 0; }

cudaError_t launch_attn_tc(const AttnProblem &p, cudaStream_t st) {
  const Plan pl = make_plan(p);
  const int group = p.hq / p.hkv;
  const int64_t cstride = (int64_t)p.seq_len * p.hkv * p.d;  // cache batch stride
  const int64_t fstride = (int64_t)p.nq * p.hkv * p.d;       // fresh batch stride
  const int64_t qstride = (int64_t)p.nq * p.hq * p.d;
  CUtensorMap maps[7];
  const __nv_bfloat16 *kc = (const __nv_bfloat16 *)p.kc, *vc = (const __nv_bfloat16 *)p.vc;
  // per-sequence blocks: prefix and suffix tiles are read through maps of the whole cache; rows of a
  // sequence's own window that fall in a boundary tile are read and weighted by exactly zero
  const bool per_seq = p.blocks != nullptr;
  const int64_t off_c = per_seq ? 0 : (int64_t)pl.f1 * p.hkv * p.d;
  const int rows_a = per_seq ? p.seq_len : pl.f0, rows_c = per_seq ? p.seq_len : p.seq_len - pl.f1;
  const int kvp = pl.kvp;
  bool ok = map4(&maps[0], p.q, p.d, p.hq, p.nq, p.batch, qstride, pl.qr) &&
            map4_kv(&maps[2], p.kf, p.d, p.hkv, p.nq, p.batch, fstride, pl.tk, kvp, false) &&
            map4_kv(&maps[5], p.vf, p.d, p.hkv, p.nq, p.batch, fstride, pl.tk, kvp, false);
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
  if (!ok) return cudaErrorInvalidValue;
  Args a;
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
