// One speculative block as a CUDA graph: gamma drafting steps through the
// trimmed head followed by the verification of the drafted tokens
// ("VocabTrim: Vocabulary Pruning for Efficient Speculative Decoding in
// LLMs", Appendix C.1, Algorithm 2: lines 4-6 draft k tokens, lines 7-14
// score and verify them).
//
// vt_block_graph_create captures the block's kernels once, with the
// programmatic-dependent-launch edges between consecutive kernels, on a
// private stream, and instantiates the graph; vt_block_graph_launch replays
// it on any stream with a single launch.  The buffers are fixed at capture:
// a replay reads whatever the input buffers hold at that time.
#include <new>

#include "vt_common.cuh"
#include "vt_internal.h"

namespace vt {
namespace {

struct BlockGraph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

size_t draft_ws(const vt_block_desc& d) {
  return align_up(vt_draft_workspace_bytes(d.B, d.H, d.K), 256);
}

// the kernels of one block, on stream s.  The hidden states are inputs of
// the block: no kernel of it writes them, and a graph launch starts only
// after everything earlier in its stream has completed, so every projection
// may stage them before its dependency wait (hidden_ready).
int record_block(const vt_block_desc& d, cudaStream_t s) {
  char* ws = static_cast<char*>(d.workspace);
  const size_t dws = draft_ws(d);
  for (int j = 0; j < d.gamma; ++j) {
    const int st = draft_step_impl(
        d.hidden + (size_t)j * d.B * d.H, d.B, d.H, d.W_trim, d.trim_ids, d.K,
        d.u_draft != nullptr ? d.u_draft + (size_t)j * d.B : nullptr, d.temperature,
        d.q + (size_t)j * d.K, (int64_t)d.gamma * d.K, d.draft_tokens + j, d.gamma,
        d.dev_status, ws, dws, s, j == 0 ? 1 : 0, 1);
    if (st != VT_OK) return st;
  }
  return vt_verify(d.target_logits, d.logits_dtype, d.B, d.gamma, d.V, d.q, d.inv_map, d.K,
                   d.draft_tokens, d.u_accept, d.u_resample, d.temperature, d.out_tokens,
                   d.out_num_accepted, d.out_accept_prob, d.dev_status + 1, ws + dws,
                   d.workspace_bytes - dws, s);
}

}  // namespace
}  // namespace vt

extern "C" size_t vt_block_workspace_bytes(int32_t B, int32_t H, int32_t K, int32_t V,
                                           int32_t gamma) {
  if (B < 1 || H < 1 || K < 1 || V < 1 || gamma < 1) return 0;
  const size_t d = vt_draft_workspace_bytes(B, H, K);
  const size_t v = vt_verify_workspace_bytes(B, gamma, V, K);
  if (d == 0 || v == 0) return 0;
  return vt::align_up(d, 256) + v;
}

extern "C" int vt_block_graph_create(const vt_block_desc* desc, void** graph) {
  using namespace vt;
  if (!desc || !graph) return VT_ERR_INVALID_ARG;
  *graph = nullptr;
  const vt_block_desc& d = *desc;
  if (d.B < 1 || d.H < 1 || d.K < 1 || d.V < 1 || d.gamma < 1 || d.K > d.V)
    return VT_ERR_INVALID_ARG;
  if (!d.hidden || !d.W_trim || !d.trim_ids || !d.target_logits || !d.q || !d.draft_tokens ||
      !d.out_tokens || !d.out_num_accepted || !d.dev_status)
    return VT_ERR_INVALID_ARG;
  if (!d.workspace || (reinterpret_cast<uintptr_t>(d.workspace) & 255)) return VT_ERR_WORKSPACE;
  if (d.workspace_bytes < vt_block_workspace_bytes(d.B, d.H, d.K, d.V, d.gamma))
    return VT_ERR_WORKSPACE;

  cudaStream_t s = nullptr;
  VT_RETURN_IF_CUDA(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
  BlockGraph* g = new (std::nothrow) BlockGraph();
  if (g == nullptr) {
    cudaStreamDestroy(s);
    return VT_ERR_CUDA;
  }
  int st = VT_OK;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    st = VT_ERR_CUDA;
  } else {
    st = record_block(d, s);  // argument errors surface here, before instantiation
    cudaGraph_t graph_captured = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s, &graph_captured);
    if (st == VT_OK && e != cudaSuccess) st = VT_ERR_CUDA;
    g->graph = graph_captured;
    if (st == VT_OK && cudaGraphInstantiate(&g->exec, g->graph, 0) != cudaSuccess)
      st = VT_ERR_CUDA;
  }
  cudaStreamDestroy(s);
  if (st != VT_OK) {
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    return st;
  }
  *graph = g;
  return VT_OK;
}

extern "C" int vt_block_graph_launch(void* graph, void* stream) {
  if (!graph) return VT_ERR_INVALID_ARG;
  auto* g = static_cast<vt::BlockGraph*>(graph);
  VT_RETURN_IF_CUDA(cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)));
  return VT_OK;
}

extern "C" int vt_block_graph_destroy(void* graph) {
  if (!graph) return VT_OK;
  auto* g = static_cast<vt::BlockGraph*>(graph);
  int st = VT_OK;
  if (g->exec && cudaGraphExecDestroy(g->exec) != cudaSuccess) st = VT_ERR_CUDA;
  if (g->graph && cudaGraphDestroy(g->graph) != cudaSuccess) st = VT_ERR_CUDA;
  delete g;
  return st;
}
