// LM head + online vocabulary reduction on the 5th-generation tensor cores.
//
// logits = h W^T for the block rows (b * B <= 512), never stored.  The grid is
// one CTA per SM, in clusters of CS = 1, 2 or 4 CTAs (CS 128-row tiles cover
// the block rows): CTA c of a cluster owns block rows [128 c, 128 c + 128),
// and cluster k of K owns the units k, k + K, k + 2K, ... of the vocabulary (a
// unit: 64 rows of W), streamed through shared memory once: every CTA of the cluster
// loads 1/CS of each W tile and multicasts it to all of them, so W leaves HBM
// once per cluster and each CTA reads only its own hidden rows.  Per CTA (256
// threads):
//   warp 0  TMA producer: its hidden-row tile (a box of the block rows rounded
//           up to 16 when one CTA holds them all, else 128 rows) and its share of
//           the W tile (64-row boxes, 128-byte swizzle, L2 evict-first) per
//           64-wide K chunk, into an S-stage ring guarded by full/empty
//           mbarriers; a stage is refilled only when every CTA of the cluster
//           has consumed it (the MMA commits arrive on all their empty barriers)
//   warp 1  TMEM owner and MMA issuer: tcgen05.mma M=128 (block rows) x
//           N=64..256 (vocabulary) x K=16, fp32 accumulator in TMEM, double
//           buffered so the epilogue of tile t overlaps the MMAs of tile t+1
//   warps 4-7 epilogue: tcgen05.ld of the accumulator (one thread per block
//           row), folded into the row's VocabStat in increasing vocabulary order
// At the end every masked row writes its VocabStat for its cluster's units to
// the partials [b * B, clusters] and arrives on a 64-bit ticket in the workspace
// (high half: this call's epoch, low half: count; a ticket left by another call
// or uninitialised memory is re-armed first, so the workspace needs no
// zeroing; the last selector re-arms the tickets for a launch that repeats this
// one's epoch, as a CUDA graph replay does).  The last min(batch, 8) CTAs to arrive wait for the rest, then merge
// the partials of their sequences' masked rows and select the unmasked
// positions (select_impl.cuh); the others exit.  No CTA ever waits for one that
// cannot be scheduled, so the launch is an ordinary (programmatic dependent) one.
//
// Every mbarrier wait is bounded; a wait that gives up records a site code in
// the device error word and sets the abort flag in every CTA of the cluster.
// Producers and MMA issuers stop at their next stage, every wait that polls the
// flag returns, each CTA waits (bounded) for its own MMAs, and after a cluster
// barrier each CTA settles the copies and MMA commits addressed to it from the
// stage counts every CTA published (settle_after_abort), so that no transfer
// of a peer reaches a CTA that has left; then a second cluster barrier, TMEM
// freed, exit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <unistd.h>

#include <atomic>
#include <chrono>

#include "common.cuh"
#include "internal.h"
#include "fp8_rule.cuh"
#include "select_impl.cuh"
#include "tc.cuh"

namespace fdllm {
namespace {

constexpr int kThreads = 256;
constexpr int kUnit = 64;        // vocabulary rows per W box
constexpr int kRowBytes = 128;   // bytes of an operand row per stage (one 128-byte swizzle atom)
// The tensor maps describe both operands as rows of kMapElemBytes-byte integers: TMA only copies
// bytes, and the 128-byte swizzle is defined on bytes, so the shared-memory tiles are the same for
// any width.  x coordinates are in these units.
constexpr int kMapElemBytes = 2;
constexpr int kMapX = kRowBytes / kMapElemBytes;   // map units per stage along a row
template <bool F8>
constexpr int kChunk = F8 ? 128 : 64;   // K elements per stage: E4M3 or bf16
constexpr int kABox = 128;       // block rows per hidden-tile (one CTA's row tile)

// Rows of the hidden-tile TMA box: the block rows rounded up to 16 when one CTA holds them all, else the
// whole 128-row tile.  (A 128-row box over a tensor of fewer than 16 rows, the rest zero-filled, slowed
// the whole W stream on GB300: 230 instead of 172 us for one sequence's 4 block rows.)  Tile rows past
// the box are never written; they only feed accumulator rows that no block row owns.
__host__ __device__ __forceinline__ int hidden_box_rows(int rows, int cs) {
  return cs == 1 && rows <= kABox ? ((rows > 16 ? rows : 16) + 15) / 16 * 16 : kABox;
}
constexpr int kMaxSelectors = 8; // CTAs that run the merge + select at the end
constexpr int kPrefetchers = 24; // first CTAs to start that warm L2 with the head of every CTA's W range
constexpr int kPrefetchBytes = 768;   // bytes of each W row of a first tile warmed in L2

struct Cfg {
  static constexpr int NV = 256;                            // vocabulary rows per tile
  static constexpr int UNITS = NV / kUnit;                  // W boxes per tile
  static constexpr int A_BYTES = kABox * kRowBytes;        // this CTA's hidden tile per stage
  static constexpr int W_BYTES = NV * kRowBytes;           // W tile per stage
  static constexpr int STAGE = A_BYTES + W_BYTES;
  static constexpr int STAGES = 4;
  static constexpr int TMEM_COLS = 512;                     // two accumulators of 256 columns
  static constexpr int SMEM = STAGES * STAGE + 1024 /*align*/ + 1024 /*barriers, flags*/;
};

struct Shared {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t accf[2];
  uint64_t acce[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  int32_t issued;     // stages issued by the producer
  int32_t consumed;   // stages consumed by the MMA issuer
  uint32_t active;    // bit m: 128-row tile m has a masked row
  int32_t arrival;    // this CTA's arrival number on the ticket (1-based, 0 on failure)
  uint8_t masked[512];
};

// Arrival number (1-based) of this CTA in epoch `e` on the ticket word; 0 if the
// ticket could not be taken.  A word from another epoch (an earlier call, or
// uninitialised memory) is first re-armed to (e, 0) by compare-and-swap on the
// value read -- one CTA wins, the others see epoch e on their next read, and
// the word never holds a stale value again during this call -- then every CTA
// counts itself with one atomic add.
// The CTA whose compare-and-swap re-arms the word also zeroes `done` (if given): no selector counts
// on it before every CTA, this one included, has arrived.
__device__ int arrive_ticket(unsigned long long *word, uint32_t e, unsigned long long *done = nullptr) {
  const unsigned long long tag = (unsigned long long)e << 32;
  for (int attempt = 0; attempt < 64; ++attempt) {
    const unsigned long long v = *(volatile unsigned long long *)word;
    if ((uint32_t)(v >> 32) != e) {
      if (atomicCAS(word, v, tag) == v && done != nullptr) atomicExch(done, 0ull);
      continue;
    }
    const unsigned long long old = atomicAdd(word, 1ull);
    if ((uint32_t)(old >> 32) == e) return (int)(uint32_t)old + 1;
  }
  return 0;
}

// Wait (bounded) until all `count` CTAs of epoch `e` have arrived.  The polling
// load has acquire semantics: the partials written before the arrivals are
// visible to this thread, and to the rest of its CTA after a __syncthreads.
__device__ bool wait_ticket(const unsigned long long *word, uint32_t e, int count) {
  const unsigned long long want = ((unsigned long long)e << 32) | (unsigned)count;
  const uint64_t t0 = tc::globaltimer();
  for (uint32_t i = 0;; ++i) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(word) : "memory");
    if (v == want) return true;
    if ((i & 63u) == 0 && tc::globaltimer() - t0 > tc::kWaitLimitNs) return false;
    __nanosleep(64);
  }
}

// A wait of this CTA gave up: record the site and stop the whole cluster.  The flag is set in
// every CTA of the cluster (distributed shared memory when CS > 1 and the launch has CS-CTA
// clusters), so every producer and MMA issuer stops at its next stage and every wait that polls the
// flag returns; the settlement after the first cluster barrier then accounts for the transfers that
// were already in flight.
template <int CS>
__device__ __forceinline__ void set_abort(Shared &sh, int32_t *err, int site, bool cluster) {
  record_device_error(err, site);
  if (CS > 1 && cluster) {
    for (uint32_t r = 0; r < (uint32_t)CS; ++r) tc::st_cluster_u32(tc::cluster_map(&sh.abort, r), 1u);
  } else {
    atomicExch(&sh.abort, 1);
  }
}

// Bytes of one stage that cluster CTA r loads into every CTA: its W boxes u = r, r + CS, ... < nu.
template <int CS>
__device__ __forceinline__ uint32_t share_bytes(int r, int nu) {
  return r < nu ? (uint32_t)((nu - r + CS - 1) / CS) * (uint32_t)(kUnit * kRowBytes) : 0u;
}

// After an abort, with every producer and MMA issuer of the cluster stopped (first cluster barrier
// passed), wait until every copy and every MMA commit addressed to this CTA has landed, so that no
// transfer reaches it after it exits.  issued[r] / consumed[r] are the stage counts of cluster CTA
// r (copies issued by its producer; stages whose MMAs its issuer committed).  A peer issues stage
// i only after its empty barrier saw every CTA's commit for stage i - STAGES, so the copies still
// unaccounted for here are those of stages [consumed[c], max issued), one use per ring slot.  Each
// such full barrier is completed exactly: bytes that a peer never sent are completed by hand
// (complete_tx), and a stage this CTA never armed is armed for the bytes the peers did send.  The
// commits are settled the same way on the empty barriers: arrivals of CTAs that never committed a
// stage are made by this CTA itself, and the phase then completes when the real ones have landed.
template <int CS>
__device__ void settle_after_abort(Shared &sh, int c, int nu_k, int kchunks, uint32_t a_bytes, int32_t *err) {
  using C = Cfg;
  int iss[CS], con[CS];
  int hi_iss = 0, hi_con = 0;
#pragma unroll
  for (int r = 0; r < CS; ++r) {
    if (CS > 1) {
      iss[r] = (int)tc::ld_cluster_u32(tc::cluster_map(&sh.issued, (uint32_t)r));
      con[r] = (int)tc::ld_cluster_u32(tc::cluster_map(&sh.consumed, (uint32_t)r));
    } else {
      iss[r] = sh.issued;
      con[r] = sh.consumed;
    }
    hi_iss = max(hi_iss, iss[r]);
    hi_con = max(hi_con, con[r]);
  }
  // copies into this CTA
  for (int it = con[c]; it < hi_iss; ++it) {
    const int st = it % C::STAGES;
    const int t = it / kchunks;
    const int nu = min(C::UNITS, nu_k - t * C::UNITS);
    uint32_t sent = iss[c] > it ? a_bytes : 0u;             // this CTA's own hidden tile
#pragma unroll
    for (int r = 0; r < CS; ++r)
      if (iss[r] > it) sent += share_bytes<CS>(r, nu);
    if (iss[c] > it) {
      const uint32_t armed = a_bytes + (uint32_t)nu * (uint32_t)(kUnit * kRowBytes);
      if (armed > sent) tc::mbar_complete_tx(&sh.full[st], armed - sent);
    } else {
      tc::mbar_arrive_expect_tx(&sh.full[st], sent);
    }
    if (!tc::mbar_wait(&sh.full[st], (uint32_t)(it / C::STAGES) & 1u)) record_device_error(err, 112);
  }
  // MMA commits into this CTA's empty barriers (its producer waited for those of stages below
  // issued[c] - STAGES)
  for (int it = max(0, iss[c] - C::STAGES); it < hi_con; ++it) {
    const int st = it % C::STAGES;
    int n = 0;
#pragma unroll
    for (int r = 0; r < CS; ++r) n += con[r] > it;
    if (n < CS) tc::mbar_arrive_count(&sh.empty[st], (uint32_t)(CS - n));
    if (!tc::mbar_wait(&sh.empty[st], (uint32_t)(it / C::STAGES) & 1u)) record_device_error(err, 113);
  }
}

// F8: E4M3 operands (the hidden rows quantised per row in the workspace, the FP8 weight cache) with
// per-row power-of-two scales h_scale [b * B] and w_scale [V]: logit = acc * h_scale * w_scale.
template <int CS, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                     const SelectProblem sp, VocabStat *__restrict__ part, unsigned long long *ticket,
                     uint32_t epoch, const float *h_scale, const float *__restrict__ w_scale) {
  constexpr int KC = kChunk<F8>;                           // K elements per stage
  const int32_t *__restrict__ tokens = sp.tokens;
  const int batch = sp.batch, seq_len = sp.seq_len, B = sp.B, mask_id = sp.mask_id, H = sp.H, V = sp.V;
  int32_t *err = sp.err;
  using C = Cfg;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *tiles = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Shared &sh = *(Shared *)(tiles + C::STAGES * C::STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = batch * B;
  const int G = gridDim.x, g = blockIdx.x;
  const int c = CS > 1 ? (int)tc::cluster_ctarank() : 0;   // this CTA's row tile
  const int ncl = G / CS, k = g / CS;                      // vocabulary splits = clusters; this cluster
  const uint32_t a_bytes = (uint32_t)(hidden_box_rows(rows, CS) * kRowBytes);   // hidden tile per stage
  constexpr uint16_t kAll = (uint16_t)((1u << CS) - 1u);   // every CTA of the cluster

  // vocabulary units of this cluster: k, k + ncl, k + 2 ncl, ... (position p of its list is unit
  // k + p ncl), so that at each step of their loops all clusters stream neighbouring rows of W: the
  // grid sweeps W in order
  const int units = (V + kUnit - 1) / kUnit;
  const int nu_k = k < units ? (units - 1 - k) / ncl + 1 : 0;
  auto unit_of = [&](int pos) { return k + pos * ncl; };
  const int ntiles = (nu_k + C::UNITS - 1) / C::UNITS;
  const int kchunks = H / KC;

  if (threadIdx.x == 0) {
    sh.abort = 0; sh.issued = 0; sh.consumed = 0; sh.active = 0;
    for (int i = 0; i < C::STAGES; ++i) {
      tc::mbar_init(&sh.full[i], 1);
      tc::mbar_init(&sh.empty[i], CS);               // one MMA commit from each CTA of the cluster
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sh.accf[i], 1);
      tc::mbar_init(&sh.acce[i], 4);
    }
    tc::mbar_init(&sh.drain, 1);
    tc::fence_barrier_init();
    tc::prefetch_tensormap(&map_h);
    tc::prefetch_tensormap(&map_w);
  }
  if (warp == 1) tc::tmem_alloc(&sh.tmem_base, C::TMEM_COLS);
  if (CS == 1 && warp == 3) {
    // The first CTAs to start usually run beside the previous kernel (programmatic dependent
    // launch, on SMs it leaves idle): they ask L2 for the first K chunks of the first W tile of
    // every CTA's range, so the main loops begin on L2 hits while HBM is otherwise little used.
    // A prefetch returns no data, so it is safe even before the previous kernel has finished.
    int e = 0;
    if (lane == 0) e = arrive_ticket(ticket + 1, epoch);
    e = __shfl_sync(0xffffffffu, e, 0);
    if (e >= 1 && e <= kPrefetchers) {
      // one W box (64 rows x 128 bytes) per prefetch: the boxes of the first kPrefetchBytes of each
      // row of the first tile of CTAs e - 1, e - 1 + kPrefetchers, ...
      const int nchunk = min(kPrefetchBytes / kRowBytes, kchunks);
      for (int j = e - 1; j < G; j += kPrefetchers) {
        const int nu = j < units ? min(C::UNITS, (units - 1 - j) / ncl + 1) : 0;
        for (int q = lane; q < nu * nchunk; q += 32)
          tc::prefetch_l2_tile_2d(&map_w, (q / nu) * kMapX, (j + (q % nu) * ncl) * kUnit);
      }
    }
  }
  // Launched as a programmatic dependent: everything above overlaps the previous kernel in the
  // stream, which may produce the tokens, hidden rows or W (or still read the workspace).
  tc::pdl_wait_primary();
  tc::pdl_launch_dependents();
  if constexpr (F8) {
    // quant_hidden: the block's hidden rows into E4M3 by the row quantiser's rule, row g by CTA g (the
    // lowest CTA indices, which wait for no one), each then arriving on the quantisation ticket; every
    // CTA waits for all of them before it reads a quantised row or scale (producer, epilogue)
    if (sp.quant_hidden && g < rows) {
      const __nv_bfloat16 *hrow = (const __nv_bfloat16 *)sp.hidden + (int64_t)g * H;
      uint8_t *qrow = (uint8_t *)sp.hq + (int64_t)g * H;
      const bool vec = H % 16 == 0 && ((uintptr_t)sp.hidden & 15) == 0 && ((uintptr_t)sp.hq & 15) == 0;
      fp8rule::quantize_row<kThreads>(hrow, H, qrow, const_cast<float *>(h_scale) + g, vec, (float *)tiles);
      if (threadIdx.x == 0) {
        __threadfence();
        if (arrive_ticket(ticket + 3, epoch) == 0) record_device_error(err, 114);
      }
    }
  }
  __syncthreads();
  // masked block rows (same on every CTA)
  for (int r = threadIdx.x; r < CS * kABox; r += kThreads) {
    bool m = false;
    if (r < rows) {
      const int bb = r / B, i = r - bb * B;
      const int sb = seq_block_start(sp, bb);
      m = sb >= 0 && tokens[(int64_t)bb * seq_len + sb + i] == mask_id;
    }
    sh.masked[r] = m;
    if (m) atomicOr(&sh.active, 1u << (r / kABox));
  }
  tc::fence_before_sync();
  if (CS > 1 && tc::cluster_nctarank() == (uint32_t)CS) tc::cluster_sync();   // barriers exist before any multicast
  else __syncthreads();
  tc::fence_after_sync();
  const uint32_t active = sh.active;
  const uint32_t tmem = sh.tmem_base;
  // The whole cluster runs the pipeline when any of its row tiles has a masked row (a CTA whose own
  // tile has none still loads its share of W and releases the stages); only masked rows are kept.
  // A launch whose clusters are not CS CTAs (never from this file's launcher) multicasts nothing:
  // it records an error and produces no partials.
  const bool shape_ok = CS == 1 || tc::cluster_nctarank() == (uint32_t)CS;
  if (!shape_ok && threadIdx.x == 0) record_device_error(err, 111);
  const bool run = shape_ok && active != 0 && ntiles > 0;
  const volatile int32_t *abort_flag = &sh.abort;       // set in every CTA of the cluster on a failure

  if (run) {
    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        const uint64_t pol_w = tc::policy_evict_first();
        const uint64_t pol_h = tc::policy_evict_last();
        int it = 0;
        bool go = true;
        if (F8 && sp.quant_hidden) {
          // every hidden row quantised (its generic writes then made visible to this thread's TMA)
          if (!wait_ticket(ticket + 3, epoch, rows)) {
            set_abort<CS>(sh, err, 115, shape_ok);
            go = false;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        for (int t = 0; t < ntiles && go; ++t) {
          const int nu = min(C::UNITS, nu_k - t * C::UNITS);
          const uint32_t bytes = a_bytes + (uint32_t)(nu * kUnit * kRowBytes);
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            const int st = it % C::STAGES;
            const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
            if (*abort_flag || !tc::mbar_wait_or_abort(&sh.empty[st], ph ^ 1u, abort_flag)) {
              if (!*abort_flag) set_abort<CS>(sh, err, 101, shape_ok);
              go = false;
              break;
            }
            unsigned char *a = tiles + st * C::STAGE;
            unsigned char *w = a + C::A_BYTES;
            tc::mbar_arrive_expect_tx(&sh.full[st], bytes);
            tc::tma_load_2d(a, &map_h, &sh.full[st], kc * kMapX, c * kABox, pol_h);
            for (int u = c; u < nu; u += CS) {
              if (CS == 1)
                tc::tma_load_2d(w + u * kUnit * kRowBytes, &map_w, &sh.full[st], kc * kMapX,
                                unit_of(t * C::UNITS + u) * kUnit, pol_w);
              else
                tc::tma_load_2d_multicast(w + u * kUnit * kRowBytes, &map_w, &sh.full[st], kc * kMapX,
                                          unit_of(t * C::UNITS + u) * kUnit, kAll, pol_w);
            }
            atomicExch(&sh.issued, it + 1);
          }
        }
        if (CS > 1 && go) {
          // every CTA of the cluster has released every stage: no commit of theirs is still on its
          // way to this CTA's barriers when it leaves (after an abort the settlement does this)
          for (int i = 0; i < C::STAGES; ++i, ++it)
            if (!tc::mbar_wait_or_abort(&sh.empty[it % C::STAGES], ((uint32_t)(it / C::STAGES) & 1u) ^ 1u,
                                        abort_flag)) {
              if (!*abort_flag) set_abort<CS>(sh, err, 110, shape_ok);
              break;
            }
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        int it = 0;
        for (int t = 0; t < ntiles && !*abort_flag; ++t) {
          const int nu = min(C::UNITS, nu_k - t * C::UNITS);
          const uint32_t idesc =
              F8 ? tc::idesc_e4m3_f32(128, (uint32_t)(nu * kUnit)) : tc::idesc_bf16_f32(128, (uint32_t)(nu * kUnit));
          const int j = t & 1;
          if (!tc::mbar_wait_or_abort(&sh.acce[j], ((uint32_t)(t >> 1) & 1u) ^ 1u, abort_flag)) {
            if (!*abort_flag) set_abort<CS>(sh, err, 102, shape_ok);
            break;
          }
          tc::fence_after_sync();
          bool ok = true;
          for (int kc = 0; kc < kchunks; ++kc, ++it) {
            const int st = it % C::STAGES;
            const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
            if (*abort_flag || !tc::mbar_wait_or_abort(&sh.full[st], ph, abort_flag)) {
              if (!*abort_flag) set_abort<CS>(sh, err, 103, shape_ok);
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t a = tc::smem_u32(tiles + st * C::STAGE);
            const uint32_t w = a + C::A_BYTES;
            const uint32_t d = tmem + (uint32_t)(j * C::NV);
#pragma unroll
            for (int kk = 0; kk < kRowBytes / 32; ++kk) {    // 32 bytes of K per instruction
              if constexpr (F8)
                tc::mma_e4m3(d, tc::sw128_desc(a + kk * 32), tc::sw128_desc(w + kk * 32), idesc, (kc | kk) != 0);
              else
                tc::mma_bf16(d, tc::sw128_desc(a + kk * 32), tc::sw128_desc(w + kk * 32), idesc, (kc | kk) != 0);
            }
            if (CS == 1) tc::mma_commit(&sh.empty[st]);
            else tc::mma_commit_multicast(&sh.empty[st], kAll);
            atomicExch(&sh.consumed, it + 1);
          }
          if (!ok) break;
          tc::mma_commit(&sh.accf[j]);
        }
        // every MMA this thread issued has completed once `drain` fires
        tc::mma_commit(&sh.drain);
        if (!tc::mbar_wait(&sh.drain, 0)) record_device_error(err, 104);
      }
    } else if (warp >= 4) {
      // ---------------- epilogue ----------------
      const int q = warp - 4;  // TMEM lane quadrant of this warp
      const int row = c * kABox + q * 32 + lane;
      const bool valid = ((active >> c) & 1) && sh.masked[row] != 0;
      const bool any = __ballot_sync(0xffffffffu, valid) != 0u;
      VocabStat st = vs_identity();
      if (F8 && sp.quant_hidden) {                     // the scales are written by other CTAs
        if (lane == 0 && !wait_ticket(ticket + 3, epoch, rows)) set_abort<CS>(sh, err, 115, shape_ok);
        __syncwarp();
      }
      const float hs = F8 && row < rows ? __ldcg(h_scale + row) : 1.f;   // this row's scale
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int ncol = min(C::UNITS, nu_k - t * C::UNITS) * kUnit;
        const int j = t & 1;
        if (!tc::mbar_wait_or_abort(&sh.accf[j], (uint32_t)(t >> 1) & 1u, abort_flag)) {
          if (lane == 0 && !*abort_flag) set_abort<CS>(sh, err, 105, shape_ok);
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (any) {
          // 32 columns at a time, reduced without branches and merged into the row's statistics (every
          // lane computes; rows without a masked position are simply not stored)
          const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(j * C::NV);
          for (int c0 = 0; c0 < ncol; c0 += 32) {
            const int vb = unit_of(t * C::UNITS + c0 / kUnit) * kUnit + c0 % kUnit;   // vocabulary id of column c0
            uint32_t r[32];
            tc::tmem_ld_32x32b_x32(base + (uint32_t)c0, r);
            // F8: lane e holds the scale of column v0 + c0 + e (both scales are powers of two, so the
            // scaled logit is exact)
            const float wsl = F8 && vb + lane < V ? __ldg(w_scale + vb + lane) : 0.f;
            tc::tmem_ld_wait();
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float a = F8 ? __uint_as_float(r[e]) * hs * __shfl_sync(0xffffffffu, wsl, e) : __uint_as_float(r[e]);
              x[e] = vb + e < V ? a : kNegInf;
            }
            st = vs_merge(st, vs_chunk32(x, vb));
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sh.acce[j]);
      }
      if (valid && row < rows) part[(int64_t)row * ncl + k] = st;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // This CTA has stopped issuing copies and MMAs, and its MMAs are complete.  After the first cluster
  // barrier every CTA of the cluster has stopped too, and an abort anywhere is visible everywhere, so
  // either no CTA or every CTA settles.
  if (CS > 1 && shape_ok) tc::cluster_sync();
  if (*abort_flag && run && threadIdx.x == 0) settle_after_abort<CS>(sh, c, nu_k, kchunks, a_bytes, err);
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, C::TMEM_COLS);
  if (CS > 1 && shape_ok) tc::cluster_sync();          // no CTA leaves while a peer may still address it

  // ---- tail: the last W CTAs to arrive select (W = min(batch, 8, grid)) ----
  // Selector w (arrival G - W + 1 + w) takes sequences w, w + W, ...  When it arrives, at most W - 1
  // CTAs have not, and the G - W CTAs that arrived before it have left their SMs, so whatever has
  // not arrived can always be scheduled: the kernel needs no co-residency guarantee.  With one
  // sequence the selector is the last CTA and never waits.
  if (threadIdx.x == 0) {
    __threadfence();                                   // this CTA's partials before its arrival
    const int a = arrive_ticket(ticket, epoch, ticket + 2);
    if (a == 0) record_device_error(err, 106);
    sh.arrival = a;
  }
  __syncthreads();
  const int W = min(min(batch, kMaxSelectors), G);
  const int sel = sh.arrival - (G - W) - 1;            // selector index, < 0 for the first G - W arrivals
  if (sh.arrival == 0 || sel < 0) return;
  SelectScratch &sc = *(SelectScratch *)tiles;         // the tile ring is free now
  // the masked positions from the flags this CTA computed at its start: the tokens are not read again
  select_prepare<kThreads>(sp, sel, sc, sh.masked);    // overlaps the wait below
  if (threadIdx.x == 0 && !wait_ticket(ticket, epoch, G)) record_device_error(err, 107);
  __syncthreads();
  select_finish<kThreads>(sp, part, ncl, sel, sc);
  for (int seq = sel + W; seq < batch; seq += W) select_sequence<kThreads>(sp, part, ncl, seq, sc, sh.masked);
  // The last selector to finish re-arms both tickets to (this epoch, 0): every CTA has arrived and
  // every selector has seen the full count, so no one reads them again in this launch.  A launch that
  // repeats this one's parameters (a CUDA graph replay: same epoch) then counts from zero.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ticket + 2, 1ull) + 1 == (unsigned long long)W) {
      const unsigned long long armed = (unsigned long long)epoch << 32;
      atomicExch(ticket, armed);
      atomicExch(ticket + 1, armed);
      atomicExch(ticket + 3, armed);
      atomicExch(ticket + 2, 0ull);
    }
  }
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

// Row-major matrix [rows, cols] of bf16 (or, with f8, E4M3 bytes) as a 2-D map of kMapElemBytes-byte
// units with box [128 bytes of a row, box_rows], 128-byte swizzle.  Row bytes are a multiple of 128.
bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows, bool f8) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t row_bytes = cols * (f8 ? 1 : 2);
  const cuuint64_t dims[2] = {row_bytes / kMapElemBytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)kMapX, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType unit = kMapElemBytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : kMapElemBytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                   : kMapElemBytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                                        : CU_TENSOR_MAP_DATA_TYPE_UINT64;
  return fn(map, unit, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int CS, bool F8>
cudaError_t launch_cs(const SelectProblem &p, VocabStat *part, unsigned long long *ticket, uint32_t epoch,
                      int splits, cudaStream_t st) {
  CUtensorMap mh, mw;
  if (!make_map(&mh, F8 ? p.hq : p.hidden, (uint64_t)p.batch * p.B, (uint64_t)p.H,
                (uint32_t)hidden_box_rows(p.batch * p.B, CS), F8) ||
      !make_map(&mw, p.w, (uint64_t)p.V, (uint64_t)p.H, kUnit, F8))
    return cudaErrorInvalidValue;
  auto kfn = lmhead_tc_kernel<CS, F8>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
  if (e != cudaSuccess) return e;
  // an ordinary launch: the tail's waiting CTAs never hold an SM that an unscheduled CTA needs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(splits * CS));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // prologue overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CS > 1 ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kfn, mh, mw, p, part, ticket, epoch, F8 ? p.h_scale : (const float *)nullptr,
                         F8 ? p.w_scale : (const float *)nullptr);
  count_launches(1);
  return e;
}

// CTAs per cluster: one per 128-row tile of block rows
int cluster_size(const SelectProblem &p) {
  const int rows = p.batch * p.B;
  return rows <= 128 ? 1 : (rows <= 256 ? 2 : 4);
}

// Clusters of CS CTAs that can be resident at once on the current device (a cluster must fit in one
// GPC, so this can be below SMs / CS); 0 if the query fails.  Cached per device.
template <int CS>
int max_active_clusters() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] > 0) return cache[dev];
  auto kfn = lmhead_tc_kernel<CS, false>;   // the E4M3 form has the same resources
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sm_count() / CS * CS));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kfn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cache[dev] = n;
  return n;
}

}  // namespace

bool lmhead_tc_supported(const SelectProblem &p) {
  return p.in_bf16 && (int64_t)p.batch * p.B <= 512 && p.H % kChunk<false> == 0 &&
         (!p.fp8w || p.H % kChunk<true> == 0);
}

bool lmhead_tc_clustered(const SelectProblem &p) { return cluster_size(p) > 1; }

// The FP8-weight LM head quantises the block's hidden rows itself when one CTA row tile holds them
// and the grid has a CTA for each (the row quantiser kernel is then not launched).
bool lmhead_tc_quantises_hidden(const SelectProblem &p) {
  return p.fp8w && cluster_size(p) == 1 && p.batch * p.B <= lmhead_tc_grid(p);
}

int lmhead_tc_grid(const SelectProblem &p) {
  // vocabulary splits = clusters: as many as can be resident at once (one CTA per SM), at least one
  // 64-row unit each
  const int units = (p.V + kUnit - 1) / kUnit;
  const int cs = cluster_size(p);
  int ncl = sm_count() / cs;
  if (cs > 1) {
    const int m = cs == 2 ? max_active_clusters<2>() : max_active_clusters<4>();
    if (m > 0 && m < ncl) ncl = m;
  }
  if (ncl < 1) ncl = 1;
  return units < ncl ? units : ncl;
}

cudaError_t launch_lmhead_tc(const SelectProblem &p, VocabStat *part, unsigned long long *ticket, int splits,
                             cudaStream_t st) {
  static std::atomic<uint32_t> epochs{(uint32_t)std::chrono::steady_clock::now().time_since_epoch().count() ^
                                      ((uint32_t)getpid() << 16)};
  uint32_t e = epochs.fetch_add(1) + 1;
  while (e == 0 || e == 0xFFFFFFFFu) e = epochs.fetch_add(1) + 1;  // never the all-zero / all-one patterns
  if (p.fp8w) {
    switch (cluster_size(p)) {
      case 1: return launch_cs<1, true>(p, part, ticket, e, splits, st);
      case 2: return launch_cs<2, true>(p, part, ticket, e, splits, st);
      default: return launch_cs<4, true>(p, part, ticket, e, splits, st);
    }
  }
  switch (cluster_size(p)) {
    case 1: return launch_cs<1, false>(p, part, ticket, e, splits, st);
    case 2: return launch_cs<2, false>(p, part, ticket, e, splits, st);
    default: return launch_cs<4, false>(p, part, ticket, e, splits, st);
  }
}

}  // namespace fdllm
