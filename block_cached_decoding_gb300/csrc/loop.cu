// Device-driven block loop.
//
// One denoising step -- whatever the caller's step function enqueues on the
// capture stream: the step's inputs, the block attention, the confidence
// select -- is captured once as the body of a CUDA graph while-loop.  A small
// control kernel ends each iteration: it counts the step in a device word and
// keeps the loop running while some sequence still has a masked position in the
// block (n_masked_left[b] > 0) and fewer than max_steps steps have run.  A
// launch therefore runs a whole block with no host round trip between steps;
// the body starts with the loop's condition set, so it runs at least once.
//
// The graph: [reset the step counter] -> [while (condition) { body }], body =
// [captured step] -> [control]; with a cache refresh every r steps (the
// refresh-every-r-steps cache variant of the summary's section 5, Table 10),
// body = [if (refresh condition) { captured refresh }] -> [captured step] ->
// [control], the control kernel setting the refresh condition for step c of
// the block when r divides c.
//
// Per-sequence blocks (the batch regime in which each sequence moves to its
// next block as soon as its own block has no mask): one loop covers the whole
// generation.  Its control kernel advances, after each step, every sequence
// whose block is done -- block index and window start in device arrays that
// the captured calls read, a refresh flag set -- or marks it finished after its
// last block; the loop runs while some sequence is unfinished, and the refresh
// node of the next iteration (the caller's refresh of the flagged sequences'
// caches) runs when some sequence advanced.
#include "common.cuh"
#include "internal.h"

struct fdllm_block_loop {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

namespace fdllm {
namespace {

__global__ void loop_reset_kernel(int64_t *counter) { *counter = 0; }

// After the step that brought the counter to c: keep looping while some sequence has a masked position
// and c < max_steps; with a refresh every r steps, arm the refresh node of the next iteration when r
// divides c (the step about to run is step c of the block, and the cache refresh comes first).
__global__ void loop_control_kernel(cudaGraphConditionalHandle cond, const int32_t *__restrict__ n_left,
                                    int batch, int64_t *counter, int64_t *total, int64_t max_steps,
                                    cudaGraphConditionalHandle refresh_cond, int64_t refresh_every) {
  __shared__ int any;
  if (threadIdx.x == 0) any = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < batch; b += blockDim.x)
    if (n_left[b] > 0) any = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t c = *counter + 1;
    *counter = c;
    if (total != nullptr) *total += 1;
    cudaGraphSetConditional(cond, any && c < max_steps ? 1u : 0u);
    if (refresh_every > 0) cudaGraphSetConditional(refresh_cond, c % refresh_every == 0 ? 1u : 0u);
  }
}

// Per-sequence blocks, after the step that brought the counter to c: each unfinished sequence counts
// the step; one whose block has no masked position moves to its next block (index, window start,
// refresh flag) or, after its last block, is finished.  Keep looping while some sequence is unfinished
// and c < max_steps; run the refresh node next iteration when some sequence moved.
__global__ void ragged_control_kernel(cudaGraphConditionalHandle cond, const int32_t *__restrict__ n_left,
                                      int batch, int nblocks, int block_size, int32_t *block_idx,
                                      int32_t *block_start, int32_t *seq_steps, uint8_t *refresh, uint8_t *done,
                                      int64_t *counter, int64_t *total, int64_t max_steps,
                                      cudaGraphConditionalHandle refresh_cond, int has_refresh) {
  __shared__ int active, moved;
  if (threadIdx.x == 0) { active = 0; moved = 0; }
  __syncthreads();
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    uint8_t adv = 0;
    if (!done[b]) {
      seq_steps[b] += 1;
      if (n_left[b] <= 0) {
        if (block_idx[b] + 1 >= nblocks) {
          done[b] = 1;
        } else {
          block_idx[b] += 1;
          block_start[b] += block_size;
          adv = 1;
        }
      }
    }
    refresh[b] = adv;
    if (adv) atomicOr(&moved, 1);
    if (!done[b]) atomicOr(&active, 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t c = *counter + 1;
    *counter = c;
    if (total != nullptr) *total += 1;
    cudaGraphSetConditional(cond, active && c < max_steps ? 1u : 0u);
    if (has_refresh) cudaGraphSetConditional(refresh_cond, moved ? 1u : 0u);
  }
}

// The per-sequence state a ragged loop's control kernel advances.
struct RaggedState {
  int nblocks, block_size;
  int32_t *block_idx, *block_start, *seq_steps;
  uint8_t *refresh, *done;
};

}  // namespace
}  // namespace fdllm

using namespace fdllm;

static fdllm_status loop_create(fdllm_block_loop **out, fdllm_step_fn step, fdllm_step_fn refresh, void *user,
                                const int32_t *n_masked_left, int32_t batch, int32_t max_steps,
                                int32_t refresh_every, int64_t *step_counter, int64_t *total_steps,
                                const RaggedState *rg = nullptr) {
  if (!out || !step || !n_masked_left || !step_counter) return FDLLM_EINVAL;
  if (batch < 1 || max_steps < 1 || refresh_every < 0) return FDLLM_EINVAL;
  if (refresh_every > 0 && !refresh) return FDLLM_EINVAL;
  const bool with_refresh = refresh_every > 0 || (rg != nullptr && refresh != nullptr);
  *out = nullptr;
  cudaGraph_t g = nullptr;
  cudaStream_t cs = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaError_t e = cudaGraphCreate(&g, 0);
  cudaGraphConditionalHandle cond = 0;
  cudaGraphNode_t reset = nullptr, wnode = nullptr;
  cudaGraph_t body = nullptr, captured = nullptr;
  if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&cond, g, 1, cudaGraphCondAssignDefault);
  if (e == cudaSuccess) {
    void *args[] = {&step_counter};
    cudaKernelNodeParams kp = {};
    kp.func = (void *)loop_reset_kernel;
    kp.gridDim = dim3(1);
    kp.blockDim = dim3(1);
    kp.kernelParams = args;
    e = cudaGraphAddKernelNode(&reset, g, nullptr, 0, &kp);
  }
  if (e == cudaSuccess) {
    cudaGraphNodeParams cp = {};
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = cond;
    cp.conditional.type = cudaGraphCondTypeWhile;
    cp.conditional.size = 1;
    e = cudaGraphAddNode(&wnode, g, &reset, nullptr, 1, &cp);
    if (e == cudaSuccess) body = cp.conditional.phGraph_out[0];
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  // with a refresh every r steps (or, per-sequence blocks, when a sequence moves on), the body starts
  // with an IF node holding the captured refresh; its condition is 0 at each launch (the caller
  // refreshes before step 0) and set by the control kernel
  cudaGraphConditionalHandle rcond = 0;
  cudaGraphNode_t ifnode = nullptr;
  if (e == cudaSuccess && with_refresh) {
    e = cudaGraphConditionalHandleCreate(&rcond, body, 0, cudaGraphCondAssignDefault);
    cudaGraph_t if_body = nullptr;
    if (e == cudaSuccess) {
      cudaGraphNodeParams ip = {};
      ip.type = cudaGraphNodeTypeConditional;
      ip.conditional.handle = rcond;
      ip.conditional.type = cudaGraphCondTypeIf;
      ip.conditional.size = 1;
      e = cudaGraphAddNode(&ifnode, body, nullptr, nullptr, 0, &ip);
      if (e == cudaSuccess) if_body = ip.conditional.phGraph_out[0];
    }
    if (e == cudaSuccess) e = cudaStreamBeginCaptureToGraph(cs, if_body, nullptr, nullptr, 0, cudaStreamCaptureModeRelaxed);
    if (e == cudaSuccess) {
      refresh(user, (fdllm_stream_t)cs);
      const cudaError_t le = cudaGetLastError();
      cudaGraph_t captured_if = nullptr;
      e = cudaStreamEndCapture(cs, &captured_if);
      if (e == cudaSuccess) e = le;
    }
  }
  if (e == cudaSuccess)
    e = cudaStreamBeginCaptureToGraph(cs, body, ifnode ? &ifnode : nullptr, nullptr, ifnode ? 1 : 0,
                                      cudaStreamCaptureModeRelaxed);
  if (e == cudaSuccess) {
    step(user, (fdllm_stream_t)cs);
    if (rg != nullptr)
      ragged_control_kernel<<<1, 256, 0, cs>>>(cond, n_masked_left, batch, rg->nblocks, rg->block_size,
                                               rg->block_idx, rg->block_start, rg->seq_steps, rg->refresh, rg->done,
                                               step_counter, total_steps, (int64_t)max_steps, rcond,
                                               with_refresh ? 1 : 0);
    else
      loop_control_kernel<<<1, 256, 0, cs>>>(cond, n_masked_left, batch, step_counter, total_steps,
                                             (int64_t)max_steps, rcond, (int64_t)refresh_every);
    const cudaError_t le = cudaGetLastError();
    e = cudaStreamEndCapture(cs, &captured);
    if (e == cudaSuccess) e = le;
  }
  if (cs) cudaStreamDestroy(cs);
  if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, g, 0);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    (void)cudaGetLastError();
    return FDLLM_ECUDA;
  }
  *out = new fdllm_block_loop{g, exec};
  return FDLLM_OK;
}

extern "C" fdllm_status fdllm_block_loop_create(fdllm_block_loop **out, fdllm_step_fn step, void *user,
                                                const int32_t *n_masked_left, int32_t batch, int32_t max_steps,
                                                int64_t *step_counter, int64_t *total_steps) {
  return loop_create(out, step, nullptr, user, n_masked_left, batch, max_steps, 0, step_counter, total_steps);
}

extern "C" fdllm_status fdllm_block_loop_create_refresh(fdllm_block_loop **out, fdllm_step_fn step,
                                                        fdllm_step_fn refresh, void *user,
                                                        const int32_t *n_masked_left, int32_t batch,
                                                        int32_t max_steps, int32_t refresh_every,
                                                        int64_t *step_counter, int64_t *total_steps) {
  if (refresh_every < 1) return FDLLM_EINVAL;
  return loop_create(out, step, refresh, user, n_masked_left, batch, max_steps, refresh_every, step_counter,
                     total_steps);
}

extern "C" fdllm_status fdllm_block_loop_create_ragged(fdllm_block_loop **out, fdllm_step_fn step,
                                                       fdllm_step_fn refresh, void *user,
                                                       const int32_t *n_masked_left, int32_t batch, int32_t n_blocks,
                                                       int32_t block_size, int32_t max_steps, int32_t *block_idx,
                                                       int32_t *block_start, int32_t *seq_steps, uint8_t *refresh_flags,
                                                       uint8_t *done, int64_t *step_counter, int64_t *total_steps) {
  if (n_blocks < 1 || block_size < 1 || !block_idx || !block_start || !seq_steps || !refresh_flags || !done)
    return FDLLM_EINVAL;
  const RaggedState rg{n_blocks, block_size, block_idx, block_start, seq_steps, refresh_flags, done};
  return loop_create(out, step, refresh, user, n_masked_left, batch, max_steps, 0, step_counter, total_steps, &rg);
}

extern "C" fdllm_status fdllm_block_loop_launch(fdllm_block_loop *loop, fdllm_stream_t stream) {
  if (!loop) return FDLLM_EINVAL;
  return cudaGraphLaunch(loop->exec, (cudaStream_t)stream) == cudaSuccess ? FDLLM_OK : FDLLM_ECUDA;
}

extern "C" void fdllm_block_loop_destroy(fdllm_block_loop *loop) {
  if (!loop) return;
  cudaGraphExecDestroy(loop->exec);
  cudaGraphDestroy(loop->graph);
  delete loop;
}
