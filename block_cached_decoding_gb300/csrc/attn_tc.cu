// Block attention on the 5th-generation tensor cores (bf16 in, fp32 accumulate).
//
// Keys are taken as three contiguous ranges, each through its own TMA map so
// that no row outside a range is ever read: the cached prefix [0, f0), the fresh
// keys of this step (nq rows, the query positions) and the cached suffix
// [f1, N).  Softmax is invariant to the order of the keys, so the key tiles of
// 128 rows are enumerated range by range and split over CTAs (split-KV).
//
// One CTA = (sequence, KV head, 128-row query tile, split of <= T key tiles):
//   warp 0     TMA: the query tile (all query heads sharing the KV head are
//              packed into the 128 rows when nq <= 128), then K and V tiles
//   warp 1     TMEM owner, MMA issuer: S_t = Q K_t^T (M=128, N=128 keys,
//              K=d) into TMEM for every tile, then O = sum_t P_t V_t
//              (N=d, K=128 keys, V read MN-major)
//   warps 4-7  one thread per query row: the row max over all the CTA's
//              scores, P_t = exp(S_t - max) written as bf16 into the
//              K_t buffer (the A operand of the second MMA, 128-byte
//              swizzled), then O / l to the output (one split) or to the
//              split-KV partials with (max, l) for the combine kernel.
// With every score tile of the CTA resident in TMEM the softmax needs a single
// max, so O never has to be rescaled.
//
// Merging the splits: when a unit has at most 8 splits they run as one thread
// block cluster and merge through distributed shared memory: every CTA
// publishes its rows' (max, l), weights its O rows by l_s 2^(m_s - M) / L and
// stores them in its own shared memory; CTA c then sums rows [c R/C, (c+1) R/C)
// across the cluster and writes the output.  Longer key ranges fall back to
// fp32 partials in the workspace and a combine kernel.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;  // keys per tile and rows per query tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxCluster = 8;  // portable thread-block cluster size

struct Plan {
  int f0, f1;           // cached prefix [0, f0), cached suffix [f1, N)
  int ka, kf, kcn;      // key tiles in the three ranges
  int kt;               // total key tiles
  int T;                // key tiles per CTA (1 or 2)
  int nsplit;
  int qr;               // query rows per head slot in a tile (multiple of 8)
  int ht;               // head slots per tile
  int qtiles_per_head;  // tiles per head when nq > 128
  int nqt;              // query tiles per KV head
  int units;            // batch * Hkv * nqt
  int cluster;          // 1: splits of a unit form a cluster and merge in DSMEM
};

template <int D>
struct Cfg {
  static constexpr int DH = D / 64;                     // 64-column halves of a row
  static constexpr int TILE_BYTES = kTile * D * 2;      // 128 rows x d bf16
  static constexpr int HALF_BYTES = kTile * 128;        // 128 rows x 64 bf16
  static constexpr int P_BYTES = kTile * kTile * 2;     // 128 rows x 128 keys bf16
  static constexpr int KP_BYTES = TILE_BYTES > P_BYTES ? TILE_BYTES : P_BYTES;  // K tile, then P
};

template <int D, int T>
struct Smem {
  static constexpr int BYTES = Cfg<D>::TILE_BYTES * (1 + T) + Cfg<D>::KP_BYTES * T + 1024 + 2048;
  static constexpr int TMEM_COLS = T == 1 ? 256 : 512;  // S tiles + O
};

struct Bars {
  uint64_t qfull, kfull[2], vfull[2], sfull[2], pfull[2], ofull, drain;
  uint32_t tmem_base;
  int32_t abort;
  float2 ml[kTile];  // this CTA's (max in log2 units, l) per row, read by the cluster
};

struct KeyTile {
  int range;   // 0 prefix cache, 1 fresh, 2 suffix cache
  int row0;    // first row within the range's map
  int nvalid;  // valid keys in the tile
};

__device__ __forceinline__ KeyTile key_tile(const Plan &pl, int nq, int n, int k) {
  KeyTile t;
  if (k < pl.ka) {
    t.range = 0; t.row0 = k * kTile; t.nvalid = min(kTile, pl.f0 - t.row0);
  } else if (k < pl.ka + pl.kf) {
    t.range = 1; t.row0 = (k - pl.ka) * kTile; t.nvalid = min(kTile, nq - t.row0);
  } else {
    t.range = 2; t.row0 = (k - pl.ka - pl.kf) * kTile; t.nvalid = min(kTile, n - pl.f1 - t.row0);
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
  float *part_o;     // [units, nsplit, 128, D] (nsplit > 1)
  float2 *part_ml;   // [units, nsplit, 128]: (max in log2 units, l)
  int32_t *err;
};

template <int D, int T, bool CL>
__global__ void __launch_bounds__(kThreads, T == 1 ? 2 : 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mka,
                   const __grid_constant__ CUtensorMap mkf, const __grid_constant__ CUtensorMap mkc,
                   const __grid_constant__ CUtensorMap mva, const __grid_constant__ CUtensorMap mvf,
                   const __grid_constant__ CUtensorMap mvc, const Args a) {
  using CF = Cfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *q_s = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char *k_s = q_s + CF::TILE_BYTES;                 // T slots: K tile, later P
  unsigned char *v_s = k_s + T * CF::KP_BYTES;               // T tiles
  Bars &br = *(Bars *)(v_s + T * CF::TILE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Plan &pl = a.pl;

  // which unit and split
  const int split = blockIdx.x % pl.nsplit;
  const int unit = blockIdx.x / pl.nsplit;
  const int qt = unit % pl.nqt;
  const int kvh = (unit / pl.nqt) % a.hkv;
  const int b = unit / (pl.nqt * a.hkv);
  const int k0 = split * T;
  const int nt = min(T, pl.kt - k0);
  // query tile: head slots [h0, h0 + nh) of the group, query rows [q0, q0 + qr)
  int h0, nh, q0;
  if (pl.qtiles_per_head == 0) {       // nq <= 128: pack heads
    h0 = qt * pl.ht; nh = min(pl.ht, a.group - h0); q0 = 0;
  } else {
    h0 = qt / pl.qtiles_per_head; nh = 1; q0 = (qt % pl.qtiles_per_head) * kTile;
  }

  if (threadIdx.x == 0) {
    br.abort = 0;
    tc::mbar_init(&br.qfull, 1);
    for (int t = 0; t < 2; ++t) {
      tc::mbar_init(&br.kfull[t], 1);
      tc::mbar_init(&br.vfull[t], 1);
      tc::mbar_init(&br.sfull[t], 1);
      tc::mbar_init(&br.pfull[t], 4);
    }
    tc::mbar_init(&br.ofull, 1);
    tc::mbar_init(&br.drain, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&br.tmem_base, Smem<D, T>::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  tc::pdl_launch_dependents();
  const uint32_t tmem = br.tmem_base;
  const uint32_t tmem_o = tmem + (uint32_t)(T * kTile);
  bool ok_cl = false;   // cluster merge: this thread's row finished its split
  float ms_cl = 0.f;    // cluster merge: this thread's row max in log2 units

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_q = tc::policy_evict_last();
      const uint64_t pol_kv = tc::policy_evict_first();
      const uint32_t qbox = (uint32_t)(pl.qr * 128);
      tc::mbar_arrive_expect_tx(&br.qfull, qbox * CF::DH * (uint32_t)nh);
      for (int hs = 0; hs < nh; ++hs)
        for (int dh = 0; dh < CF::DH; ++dh)
          tc::tma_load_4d(q_s + dh * CF::HALF_BYTES + hs * pl.qr * 128, &mq, &br.qfull, dh * 64,
                          kvh * a.group + h0 + hs, q0, b, pol_q);
      for (int t = 0; t < nt; ++t) {
        const KeyTile kt = key_tile(pl, a.nq, a.n, k0 + t);
        const CUtensorMap *mk = kt.range == 0 ? &mka : (kt.range == 1 ? &mkf : &mkc);
        const CUtensorMap *mv = kt.range == 0 ? &mva : (kt.range == 1 ? &mvf : &mvc);
        tc::mbar_arrive_expect_tx(&br.kfull[t], (uint32_t)CF::TILE_BYTES);
        for (int dh = 0; dh < CF::DH; ++dh)
          tc::tma_load_4d(k_s + t * CF::KP_BYTES + dh * CF::HALF_BYTES, mk, &br.kfull[t], dh * 64, kvh, kt.row0, b,
                          pol_kv);
        tc::mbar_arrive_expect_tx(&br.vfull[t], (uint32_t)CF::TILE_BYTES);
        for (int dh = 0; dh < CF::DH; ++dh)
          tc::tma_load_4d(v_s + t * CF::TILE_BYTES + dh * CF::HALF_BYTES, mv, &br.vfull[t], dh * 64, kvh, kt.row0, b,
                          pol_kv);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_bf16_f32(128, kTile, 0);
      const uint32_t id_o = tc::idesc_bf16_f32(128, D, 1);
      bool ok = tc::mbar_wait(&br.qfull, 0);
      if (!ok) { record_device_error(a.err, 201); atomicExch(&br.abort, 1); }
      const uint32_t qa = tc::smem_u32(q_s);
      for (int t = 0; t < nt && ok; ++t) {
        if (!tc::mbar_wait(&br.kfull[t], 0)) { record_device_error(a.err, 202); atomicExch(&br.abort, 1); ok = false; break; }
        tc::fence_after_sync();
        const uint32_t ka = tc::smem_u32(k_s + t * CF::KP_BYTES);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (uint32_t)((ks / 4) * CF::HALF_BYTES + (ks % 4) * 32);
          tc::mma_bf16(tmem + (uint32_t)(t * kTile), tc::sw128_desc(qa + off), tc::sw128_desc(ka + off), id_s, ks != 0);
        }
        tc::mma_commit(&br.sfull[t]);
      }
      for (int t = 0; t < nt && ok; ++t) {
        if (!tc::mbar_wait(&br.pfull[t], 0) || !tc::mbar_wait(&br.vfull[t], 0)) {
          record_device_error(a.err, 203); atomicExch(&br.abort, 1); ok = false; break;
        }
        tc::fence_after_sync();
        const uint32_t pa = tc::smem_u32(k_s + t * CF::KP_BYTES);
        const uint32_t va = tc::smem_u32(v_s + t * CF::TILE_BYTES);
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const uint32_t poff = (uint32_t)((ks / 4) * (kTile * 128) + (ks % 4) * 32);
          tc::mma_bf16(tmem_o, tc::sw128_desc(pa + poff), tc::sw128_mn_desc(va + (uint32_t)(ks * 2048), CF::HALF_BYTES),
                       id_o, (t | ks) != 0);
        }
      }
      if (ok) tc::mma_commit(&br.ofull);
      tc::mma_commit(&br.drain);
      if (!tc::mbar_wait(&br.drain, 0)) record_device_error(a.err, 204);
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    const int r = q * 32 + lane;                    // query row of the tile (TMEM lane)
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    bool ok = true;
    // pass 1: the row max over all valid scores of the CTA (TMEM read 64 columns per wait)
    float mx = kNegInf;
    for (int t = 0; t < nt && ok; ++t) {
      if (!tc::mbar_wait(&br.sfull[t], 0)) { record_device_error(a.err, 205); atomicExch(&br.abort, 1); ok = false; break; }
      tc::fence_after_sync();
      const int nv = key_tile(pl, a.nq, a.n, k0 + t).nvalid;
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 64) {
        uint32_t x[32], y[32];
        tc::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)(t * kTile + c0), x);
        tc::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)(t * kTile + c0 + 32), y);
        tc::tmem_ld_wait();
        if (nv >= kTile) {
#pragma unroll
          for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fmaxf(__uint_as_float(x[e]), __uint_as_float(y[e])));
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (c0 + e < nv) mx = fmaxf(mx, __uint_as_float(x[e]));
            if (c0 + 32 + e < nv) mx = fmaxf(mx, __uint_as_float(y[e]));
          }
        }
      }
    }
    // pass 2: P = exp2((s - max) * scale * log2 e) as bf16 into the K buffer; l = sum P
    float l = 0.f;
    const float ms = mx * a.scale_log2;
    for (int t = 0; t < nt && ok; ++t) {
      const int nv = key_tile(pl, a.nq, a.n, k0 + t).nvalid;
      unsigned char *p_s = k_s + t * CF::KP_BYTES;
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 64) {
        uint32_t x[64];
        tc::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)(t * kTile + c0), *(uint32_t(*)[32])&x[0]);
        tc::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)(t * kTile + c0 + 32), *(uint32_t(*)[32])&x[32]);
        tc::tmem_ld_wait();
        // these 64 keys are one 128-byte row of the swizzle atom column c0 / 64: 8 chunks of 8 keys
        unsigned char *rowp = p_s + (c0 / 64) * (kTile * 128) + r * 128;
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t pk[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int e = ch * 8 + e2 * 2;
            const float p0 = (c0 + e < nv) ? tc::ex2_approx(fmaf(__uint_as_float(x[e]), a.scale_log2, -ms)) : 0.f;
            const float p1 = (c0 + e + 1 < nv) ? tc::ex2_approx(fmaf(__uint_as_float(x[e + 1]), a.scale_log2, -ms)) : 0.f;
            l0 += p0;
            l1 += p1;
            __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
            pk[e2] = *(uint32_t *)&h2;
          }
          *(uint4 *)(rowp + ((ch ^ (r & 7)) * 16)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l += l0 + l1;
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&br.pfull[t]);
    }
    if (ok && !tc::mbar_wait(&br.ofull, 0)) { record_device_error(a.err, 206); atomicExch(&br.abort, 1); ok = false; }
    if constexpr (CL) {
      // publish this split's (max, l) of row r; O is weighted after the cluster barrier
      br.ml[r] = ok ? make_float2(ms, l) : make_float2(kNegInf, 0.f);
      ok_cl = ok;
      ms_cl = ms;
    } else if (ok) {
      tc::fence_after_sync();
      // row r of the tile -> (head, query); O streams from TMEM 32 columns at a time
      const int hs = pl.qtiles_per_head == 0 ? r / pl.qr : 0;
      const int qi = pl.qtiles_per_head == 0 ? r % pl.qr : q0 + r;
      const bool valid = hs < nh && qi < a.nq;
      const int h = kvh * a.group + h0 + hs;
      const float inv = 1.f / l;
      const int64_t obase = (((int64_t)b * a.nq + qi) * a.hq + h) * D;
      const int64_t slot = ((int64_t)unit * pl.nsplit + split) * kTile + r;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t x[32];
        tc::tmem_ld_32x32b_x32(tmem_o + lane_base + (uint32_t)c0, x);
        tc::tmem_ld_wait();
        if (!valid) continue;
        if (pl.nsplit > 1 || a.out_f32) {
          float4 *dst = pl.nsplit > 1 ? (float4 *)(a.part_o + slot * D + c0) : (float4 *)((float *)a.out + obase + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(x[4 * i]) * inv, __uint_as_float(x[4 * i + 1]) * inv,
                                 __uint_as_float(x[4 * i + 2]) * inv, __uint_as_float(x[4 * i + 3]) * inv);
        } else {
          uint4 *dst = (uint4 *)((__nv_bfloat16 *)a.out + obase + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(x[8 * i + 2 * e]) * inv,
                                                        __uint_as_float(x[8 * i + 2 * e + 1]) * inv);
              w[e] = *(uint32_t *)&h2;
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (valid) {
        if (pl.nsplit > 1)
          a.part_ml[slot] = make_float2(ms, l);
        else if (a.lse)
          a.lse[((int64_t)b * a.nq + qi) * a.hq + h] = mx * a.scale + __logf(l);
      }
    }
  }
  if constexpr (CL) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = pl.nsplit;
    const int crank = (int)cluster.block_rank();
    constexpr int CH = D / 4;                          // float4 chunks per row
    float *ored = (float *)k_s;                        // [128][D] fp32, chunks swizzled by row
    tc::fence_before_sync();
    cluster.sync();                                    // every split's (max, l) is published
    float M = kNegInf, L = 0.f;
    const int r = (warp - 4) * 32 + lane;
    if (warp >= 4) {
      tc::fence_after_sync();
      for (int c = 0; c < C; ++c) M = fmaxf(M, cluster.map_shared_rank(&br.ml[r], c)->x);
      for (int c = 0; c < C; ++c) {
        const float2 v = *cluster.map_shared_rank(&br.ml[r], c);
        if (v.y > 0.f) L += v.y * exp2f(v.x - M);
      }
      const float w = (ok_cl && L > 0.f) ? exp2f(ms_cl - M) / L : 0.f;
      const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t x[32];
        tc::tmem_ld_32x32b_x32(tmem_o + lane_base + (uint32_t)c0, x);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ch = c0 / 4 + i;
          float4 v = ok_cl ? make_float4(__uint_as_float(x[4 * i]) * w, __uint_as_float(x[4 * i + 1]) * w,
                                         __uint_as_float(x[4 * i + 2]) * w, __uint_as_float(x[4 * i + 3]) * w)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          *(float4 *)(ored + r * D + ((ch ^ (r & (CH - 1))) * 4)) = v;
        }
      }
    }
    tc::fence_before_sync();
    cluster.sync();                                    // every split's weighted O is in its shared memory
    // this CTA sums rows [r0, r1) over the cluster and writes them
    const int rpc = (kTile + C - 1) / C;
    const int r0 = crank * rpc, r1 = min(kTile, r0 + rpc);
    for (int u = threadIdx.x; u < (r1 - r0) * CH; u += kThreads) {
      const int row = r0 + u / CH, ch = u % CH;
      const int hs = pl.qtiles_per_head == 0 ? row / pl.qr : 0;
      const int qi = pl.qtiles_per_head == 0 ? row % pl.qr : q0 + row;
      if (hs >= nh || qi >= a.nq) continue;
      const float *src = ored + row * D + ((ch ^ (row & (CH - 1))) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = 0; c < C; ++c) {
        const float4 v = *(const float4 *)cluster.map_shared_rank(src, c);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const int h = kvh * a.group + h0 + hs;
      const int64_t o = (((int64_t)b * a.nq + qi) * a.hq + h) * D + ch * 4;
      if (a.out_f32) {
        *(float4 *)((float *)a.out + o) = acc;
      } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        *(uint2 *)((__nv_bfloat16 *)a.out + o) = make_uint2(*(uint32_t *)&lo, *(uint32_t *)&hi);
      }
    }
    if (warp >= 4 && a.lse && r >= r0 && r < r1 && L > 0.f) {
      const int hs = pl.qtiles_per_head == 0 ? r / pl.qr : 0;
      const int qi = pl.qtiles_per_head == 0 ? r % pl.qr : q0 + r;
      if (hs < nh && qi < a.nq)
        a.lse[((int64_t)b * a.nq + qi) * a.hq + kvh * a.group + h0 + hs] = (M + log2f(L)) * 0.6931471805599453f;
    }
    cluster.sync();                                    // no CTA leaves while a peer reads its shared memory
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (br.abort && threadIdx.x == 0) {
    // loads issued but not consumed still land in shared memory: wait for them (bounded)
    tc::mbar_wait(&br.qfull, 0);
    for (int t = 0; t < nt; ++t) {
      tc::mbar_wait(&br.kfull[t], 0);
      tc::mbar_wait(&br.vfull[t], 0);
    }
  }
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, Smem<D, T>::TMEM_COLS);
}

// Combine the split-KV partials of each query row: one warp per (unit, row).
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const Args a) {
  tc::pdl_wait_primary();
  const Plan &pl = a.pl;
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)pl.units * kTile) return;
  const int r = (int)(wid % kTile);
  const int unit = (int)(wid / kTile);
  const int qt = unit % pl.nqt;
  const int kvh = (unit / pl.nqt) % a.hkv;
  const int b = unit / (pl.nqt * a.hkv);
  int h0, nh, q0;
  if (pl.qtiles_per_head == 0) {
    h0 = qt * pl.ht; nh = min(pl.ht, a.group - h0); q0 = 0;
  } else {
    h0 = qt / pl.qtiles_per_head; nh = 1; q0 = (qt % pl.qtiles_per_head) * kTile;
  }
  const int hs = pl.qtiles_per_head == 0 ? r / pl.qr : 0;
  const int qi = pl.qtiles_per_head == 0 ? r % pl.qr : q0 + r;
  if (hs >= nh || qi >= a.nq) return;
  const int h = kvh * a.group + h0 + hs;
  const int64_t slot0 = (int64_t)unit * pl.nsplit * kTile + r;
  float m = kNegInf;
  for (int s = 0; s < pl.nsplit; ++s) m = fmaxf(m, a.part_ml[slot0 + (int64_t)s * kTile].x);
  float L = 0.f;
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
  for (int s = 0; s < pl.nsplit; ++s) {
    const int64_t slot = slot0 + (int64_t)s * kTile;
    const float2 ml = a.part_ml[slot];
    const float w = ml.y * exp2f(ml.x - m);
    L += w;
    const float *po = a.part_o + slot * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] += w * po[lane + 32 * i];
  }
  const float inv = 1.f / L;
  const int64_t base = (((int64_t)b * a.nq + qi) * a.hq + h) * D;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    if (a.out_f32)
      ((float *)a.out)[base + lane + 32 * i] = acc[i] * inv;
    else
      ((__nv_bfloat16 *)a.out)[base + lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
  }
  if (a.lse && lane == 0) a.lse[((int64_t)b * a.nq + qi) * a.hq + h] = (m + log2f(L)) * 0.6931471805599453f;
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

Plan make_plan(const AttnProblem &p) {
  Plan pl;
  pl.f0 = p.fresh0;
  pl.f1 = p.fresh0 + p.nq;
  pl.ka = (pl.f0 + kTile - 1) / kTile;
  pl.kf = (p.nq + kTile - 1) / kTile;
  pl.kcn = (p.seq_len - pl.f1 + kTile - 1) / kTile;
  pl.kt = pl.ka + pl.kf + pl.kcn;
  const int group = p.hq / p.hkv;
  if (p.nq <= kTile) {
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
  pl.units = p.batch * p.hkv * pl.nqt;
  // key tiles per CTA: T = 1 fits two CTAs per SM; pick the smaller makespan in tile-times
  const int sms = sm_count();
  int best_t = 1;
  int64_t best = -1;
  for (int t = 1; t <= 2; ++t) {
    const int64_t ctas = (int64_t)pl.units * ((pl.kt + t - 1) / t);
    const int64_t slots = (int64_t)sms * (t == 1 ? 2 : 1);
    const int64_t cost = (ctas + slots - 1) / slots * t;
    if (best < 0 || cost < best) { best = cost; best_t = t; }
  }
  pl.T = best_t;
  pl.nsplit = (pl.kt + pl.T - 1) / pl.T;
  if (pl.nsplit > kMaxCluster) {           // long key ranges: two tiles per CTA before anything else
    pl.T = 2;
    pl.nsplit = (pl.kt + 1) / 2;
  }
  pl.cluster = pl.nsplit > 1 && pl.nsplit <= kMaxCluster;
  return pl;
}

template <int D, int T, bool CL>
cudaError_t launch_dtc(const Plan &pl, const CUtensorMap *maps, const Args &a, cudaStream_t st) {
  auto k = attn_tc_kernel<D, T, CL>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D, T>::BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.units * pl.nsplit));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<D, T>::BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL ? (unsigned)pl.nsplit : 1u;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], a);
  count_launches(1);
  return e;
}

template <int D, int T>
cudaError_t launch_dt(const AttnProblem &p, const Plan &pl, const CUtensorMap *maps, const Args &a, cudaStream_t st) {
  cudaError_t e = pl.cluster ? launch_dtc<D, T, true>(pl, maps, a, st) : launch_dtc<D, T, false>(pl, maps, a, st);
  if (e != cudaSuccess || pl.nsplit == 1 || pl.cluster) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((int64_t)pl.units * kTile + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_combine_kernel<D>, a);
  count_launches(1);
  return e;
}

}  // namespace

bool attn_tc_supported(const AttnProblem &p) { return p.in_bf16 && (p.d == 64 || p.d == 128); }

size_t attn_tc_workspace(const AttnProblem &p) {
  const Plan pl = make_plan(p);
  if (pl.nsplit == 1 || pl.cluster) return 0;
  const size_t slots = (size_t)pl.units * pl.nsplit * kTile;
  return slots * p.d * 4 + slots * 8 + 256;
}

cudaError_t launch_attn_tc(const AttnProblem &p, cudaStream_t st) {
  const Plan pl = make_plan(p);
  const int group = p.hq / p.hkv;
  const int64_t cstride = (int64_t)p.seq_len * p.hkv * p.d;  // cache batch stride
  const int64_t fstride = (int64_t)p.nq * p.hkv * p.d;       // fresh batch stride
  const int64_t qstride = (int64_t)p.nq * p.hq * p.d;
  CUtensorMap maps[7];
  const __nv_bfloat16 *kc = (const __nv_bfloat16 *)p.kc, *vc = (const __nv_bfloat16 *)p.vc;
  const int64_t off_c = (int64_t)pl.f1 * p.hkv * p.d;
  if (!map4(&maps[0], p.q, p.d, p.hq, p.nq, p.batch, qstride, pl.qr) ||
      !map4(&maps[1], p.kc, p.d, p.hkv, pl.f0, p.batch, cstride, kTile) ||
      !map4(&maps[2], p.kf, p.d, p.hkv, p.nq, p.batch, fstride, kTile) ||
      !map4(&maps[3], kc + off_c, p.d, p.hkv, p.seq_len - pl.f1, p.batch, cstride, kTile) ||
      !map4(&maps[4], p.vc, p.d, p.hkv, pl.f0, p.batch, cstride, kTile) ||
      !map4(&maps[5], p.vf, p.d, p.hkv, p.nq, p.batch, fstride, kTile) ||
      !map4(&maps[6], vc + off_c, p.d, p.hkv, p.seq_len - pl.f1, p.batch, cstride, kTile))
    return cudaErrorInvalidValue;
  Args a;
  a.pl = pl;
  a.batch = p.batch; a.n = p.seq_len; a.nq = p.nq; a.hq = p.hq; a.hkv = p.hkv; a.group = group;
  a.scale = p.scale;
  a.scale_log2 = p.scale * kLog2e;
  a.out_f32 = p.out_f32;
  a.out = p.out;
  a.lse = p.lse;
  const size_t slots = (size_t)pl.units * pl.nsplit * kTile;
  a.part_o = (float *)p.ws;
  a.part_ml = (float2 *)((char *)p.ws + slots * p.d * 4);
  a.err = p.err;
  if (p.d == 128) return pl.T == 1 ? launch_dt<128, 1>(p, pl, maps, a, st) : launch_dt<128, 2>(p, pl, maps, a, st);
  return pl.T == 1 ? launch_dt<64, 1>(p, pl, maps, a, st) : launch_dt<64, 2>(p, pl, maps, a, st);
}

}  // namespace fdllm
