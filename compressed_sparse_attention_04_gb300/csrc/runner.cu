// Stage 5: Full / Reindex / Reuse layer runtime (host code; launches the stage kernels).
//
// [P1] "DeepSeek-V4.1 模型结构（2）：序列维度（中），CSA2 的三种模式" (blog.javazero.top):
//      §一层全局注意力算四样东西 -- a layer may take main KV, indexer K and top-k from an
//      earlier layer, only the attention is always its own; own KV with a foreign index
//      is meaningless; the mode of each layer is static config.
//      §共享池里有四样东西 -- one shared object with four single-position slots
//      (compress_kv, index_k, topk_idxs, candidates); a Full layer repoints compress_kv,
//      an index source overwrites topk_idxs; layers run in order.
//      §40 层只有 4 个 Full -- the tables kv_source_layer_ids / index_source_layer_ids.
// [P2] "DeepSeek v4.1 Flash技术剖析——架构篇" (myhz0606.com) §CSA2-ReIndex (pool built by
//      the preceding Full layer), §CSA2-Reuse.
// [P4] "CSA2 — l'attention creuse compressée de seconde génération" (mkdocs.reaper.mx)
//      §Les trois modes.
#include <memory>
#include <new>
#include <vector>

#include "common.cuh"

struct csa2_runner {
  int n_layers = 0;
  std::vector<int> kv_src, idx_src, ratio, mode;
  std::vector<char> builds_pool;
  int hsi_blk = 64, hsi_nb = 64;
  void* const* events = nullptr;   // optional per-stage timing events
  int n_events = 0;
};

namespace csa2 {
namespace {

struct WsLayout {
  size_t gemm, kv_pre, scores, blockmax, topk, cand, attn, total;
};

WsLayout layout(const csa2_runner* r, const csa2_step_params* p, int max_x_tokens, int max_entries) {
  WsLayout w{};
  const size_t rows = size_t(p->B) * p->Tq;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  const size_t gemm_bytes = csa2_compress_workspace_size(p->B, max_x_tokens > 0 ? max_x_tokens : 1, p->hidden, 2);
  w.gemm = take(gemm_bytes);
  w.kv_pre = take(size_t(p->B) * (max_x_tokens > 0 ? max_x_tokens : 1) * 512 * sizeof(float));
  // indexer scratch (scores + top-k candidate lists): the larger of a Full call over
  // max_entries and a Reindex call over the candidate pool
  const size_t full_ws = csa2_indexer_workspace_size(p->B, p->Tq, max_entries, 0, r->hsi_blk, 0);
  const size_t pool_ws = csa2_indexer_workspace_size(p->B, p->Tq, max_entries, r->hsi_nb, r->hsi_blk, 1);
  (void)rows;
  w.scores = take(full_ws > pool_ws ? full_ws : pool_ws);
  w.blockmax = take(rows * size_t(ceil_div(max_entries, r->hsi_blk)) * sizeof(float));
  w.topk = take(rows * size_t(p->k) * sizeof(int32_t));
  w.cand = take(rows * size_t(r->hsi_nb) * sizeof(int32_t));
  w.attn = take(csa2_sparse_attn_workspace_size(p->B, p->Tq, p->H, p->k, p->window));
  w.total = off;
  return w;
}

cudaEvent_t stage_event(const csa2_runner* r, int layer, int stage, int end) {
  if (!r->events) return nullptr;
  const int i = (layer * CSA2_STAGES + stage) * 2 + end;
  return i < r->n_events ? static_cast<cudaEvent_t>(r->events[i]) : nullptr;
}

void mark(const csa2_runner* r, int layer, int stage, int end, void* stream) {
  cudaEvent_t e = stage_event(r, layer, stage, end);
  if (e) record_stage_event(e, static_cast<cudaStream_t>(stream));
}

int check_params(const csa2_step_params* p) {
  if (!p) return fail(CSA2_ERR_INVALID_ARG, "runner: null params");
  if (p->B <= 0 || p->Tq <= 0 || p->q_pos0 < 0 || p->H <= 0 || p->hidden <= 0 || p->k < 1 ||
      p->k > CSA2_MAX_TOPK || p->window < 1)
    return fail(CSA2_ERR_INVALID_ARG, "runner: bad step params");
  return CSA2_OK;
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

int csa2_runner_create(int n_layers, const int32_t* kv_src, const int32_t* idx_src,
                       const int32_t* ratio, int hsi_blk, int hsi_nb, csa2_runner** out) {
  if (!out) return fail(CSA2_ERR_INVALID_ARG, "runner_create: null out");
  *out = nullptr;
  if (n_layers <= 0 || n_layers > 4096 || !kv_src || !idx_src || !ratio)
    return fail(CSA2_ERR_INVALID_ARG, "runner_create: bad table arguments");
  if (!is_pow2(hsi_blk) || hsi_blk > 256 || hsi_nb < 1 || hsi_nb > CSA2_MAX_TOPK)
    return fail(CSA2_ERR_UNSUPPORTED, "runner_create: hsi_blk=%d (power of two <= 256), hsi_nb=%d",
                hsi_blk, hsi_nb);
  std::unique_ptr<csa2_runner> r(new (std::nothrow) csa2_runner);
  if (!r) return fail(CSA2_ERR_INVALID_ARG, "runner_create: out of host memory");
  r->n_layers = n_layers;
  r->hsi_blk = hsi_blk;
  r->hsi_nb = hsi_nb;
  r->kv_src.assign(kv_src, kv_src + n_layers);
  r->idx_src.assign(idx_src, idx_src + n_layers);
  r->ratio.assign(ratio, ratio + n_layers);
  r->mode.assign(n_layers, -1);
  r->builds_pool.assign(n_layers, 0);
  for (int l = 0; l < n_layers; ++l) {
    const int f = r->kv_src[l], x = r->idx_src[l];
    if (f == -1) {
      if (x != -1) return fail(CSA2_ERR_INVALID_ARG, "layer %d: index source without a KV source", l);
      r->mode[l] = CSA2_MODE_SWA;
    } else if (f == l) {
      if (x != l) return fail(CSA2_ERR_INVALID_ARG, "layer %d: own KV with a foreign index", l);
      if (r->ratio[l] != 1 && r->ratio[l] != 2)
        return fail(CSA2_ERR_UNSUPPORTED, "layer %d: compression ratio %d (1 or 2)", l, r->ratio[l]);
      r->mode[l] = CSA2_MODE_FULL;
    } else if (f >= 0 && f < l && r->mode[f] == CSA2_MODE_FULL) {
      if (x == l) {
        r->mode[l] = CSA2_MODE_REINDEX;
        r->builds_pool[f] = 1;
      } else if (x >= 0 && x < l && (r->mode[x] == CSA2_MODE_FULL || r->mode[x] == CSA2_MODE_REINDEX) &&
                 r->kv_src[x] == f) {
        r->mode[l] = CSA2_MODE_REUSE;
      } else {
        return fail(CSA2_ERR_INVALID_ARG, "layer %d: index source %d invalid for KV source %d", l, x, f);
      }
    } else {
      return fail(CSA2_ERR_INVALID_ARG, "layer %d: KV source %d is not an earlier Full layer", l, f);
    }
  }
  *out = r.release();
  return CSA2_OK;
}

void csa2_runner_destroy(csa2_runner* r) { delete r; }

int csa2_runner_set_timing(csa2_runner* r, void* const* events, int n_events) {
  if (!r) return fail(CSA2_ERR_INVALID_ARG, "runner_set_timing: null runner");
  if (events && n_events < 0) return fail(CSA2_ERR_INVALID_ARG, "runner_set_timing: n_events < 0");
  r->events = events;
  r->n_events = events ? n_events : 0;
  return CSA2_OK;
}

int csa2_runner_layer_mode(const csa2_runner* r, int layer) {
  if (!r || layer < 0 || layer >= r->n_layers) return -1;
  return r->mode[layer];
}

size_t csa2_runner_workspace_size(const csa2_runner* r, const csa2_step_params* p, int max_x_tokens,
                                  int max_entries) {
  if (!r || check_params(p) != CSA2_OK || max_x_tokens < 0 || max_entries < 0) return 0;
  return layout(r, p, max_x_tokens, max_entries).total;
}

int csa2_runner_step(csa2_runner* r, const csa2_step_params* p, const csa2_layer_io* io,
                     void* workspace, size_t ws_bytes, void* stream) {
  if (!r || !io) return fail(CSA2_ERR_INVALID_ARG, "runner_step: null runner or io");
  int st = check_params(p);
  if (st != CSA2_OK) return st;
  // sizes needed by this step
  int max_x = 0, max_n = 0;
  for (int l = 0; l < r->n_layers; ++l) {
    if (r->mode[l] != CSA2_MODE_FULL) continue;
    const csa2_layer_io& L = io[l];
    if (L.x_tokens < 0 || L.x_pos0 < 0) return fail(CSA2_ERR_INVALID_ARG, "layer %d: bad x range", l);
    if (L.x_tokens > max_x) max_x = L.x_tokens;
    const int n = (L.x_pos0 + L.x_tokens) / r->ratio[l];
    if (n > max_n) max_n = n;
  }
  const WsLayout w = layout(r, p, max_x, max_n);
  if (!workspace || ws_bytes < w.total || !aligned256(workspace))
    return fail(CSA2_ERR_WORKSPACE, "runner_step: workspace needs %zu bytes, 256-aligned", w.total);
  char* ws = static_cast<char*>(workspace);
  const size_t gemm_bytes = w.kv_pre - w.gemm;

  // the four shared slots
  int slot_kv = -1;                // layer whose main KV / indexer K is current
  const int32_t* slot_topk = nullptr;
  int slot_topk_layer = -1;        // index source whose top-k is current
  const int32_t* slot_cand = nullptr;
  std::vector<int> n_entries(r->n_layers, 0);

  for (int l = 0; l < r->n_layers; ++l) {
    const csa2_layer_io& L = io[l];
    const int md = r->mode[l];
    if (md == CSA2_MODE_FULL) {
      const int m = r->ratio[l];
      if (L.x_tokens > 0) {
        mark(r, l, 0, 0, stream);
        // entries completed by this step's tokens: e0 .. e0 + g_new - 1 (with the group state a
        // step may start or end inside a group; without it, only whole groups count)
        const int e0 = L.x_pos0 / m;
        const int g_new = L.compress_state ? (L.x_pos0 + L.x_tokens) / m - e0 : L.x_tokens / m;
        // decode-sized calls write the indexer keys from the compressor's epilogue
        if (!L.w_ik || !L.idx_codes || !L.idx_scales)
          return fail(CSA2_ERR_INVALID_ARG, "layer %d: Full layer needs w_ik and the indexer-key caches", l);
        bool idx_done = false;
        st = compress_index_k(L.x, p->B, L.x_tokens, p->hidden, m, L.x_pos0, L.w_kv, L.w_gate,
                              L.norm_w, p->eps, p->rope_base, L.compress_state, L.kv_cache, L.n_cap,
                              reinterpret_cast<float*>(ws + w.kv_pre), ws + w.gemm, gemm_bytes,
                              L.w_ik, L.idx_codes, L.idx_scales, stream, &idx_done);
        if (st != CSA2_OK) return st;
        if (L.kv_codes || L.kv_scales) {   // the new entries in the stored FP4 format too
          if (!L.kv_codes || !L.kv_scales)
            return fail(CSA2_ERR_INVALID_ARG, "layer %d: FP4 main KV needs codes and scales", l);
          st = csa2_main_kv_quant_fp4(L.kv_cache, p->B, L.n_cap, e0, g_new, L.kv_codes, L.kv_scales,
                                      stream);
          if (st != CSA2_OK) return st;
        }
        mark(r, l, 0, 1, stream);
        mark(r, l, 1, 0, stream);
        if (!idx_done) {
          st = csa2_index_k_quant(reinterpret_cast<float*>(ws + w.kv_pre), p->B, g_new, e0, m, L.w_ik,
                                  p->rope_base, L.idx_codes, L.idx_scales, L.n_cap, nullptr, stream);
          if (st != CSA2_OK) return st;
        }
        mark(r, l, 1, 1, stream);
      }
      n_entries[l] = (L.x_pos0 + L.x_tokens) / m;
      slot_kv = l;
    }
    if (md == CSA2_MODE_FULL || md == CSA2_MODE_REINDEX) {
      const int f = (md == CSA2_MODE_FULL) ? l : r->kv_src[l];
      const csa2_layer_io& F = io[f];
      int32_t* topk = L.topk_out ? L.topk_out : reinterpret_cast<int32_t*>(ws + w.topk);
      const bool pool = md == CSA2_MODE_FULL && r->builds_pool[l];
      float* bmax = pool ? reinterpret_cast<float*>(ws + w.blockmax) : nullptr;
      const int32_t* cand = (md == CSA2_MODE_REINDEX) ? slot_cand : nullptr;
      if (md == CSA2_MODE_REINDEX && (!cand || slot_kv != f))
        return fail(CSA2_ERR_INVALID_ARG, "layer %d: no candidate pool from Full layer %d", l, f);
      mark(r, l, 2, 0, stream);
      st = indexer_impl(L.q_idx, L.w_idx, p->B, p->Tq, p->q_pos0, F.idx_codes, F.idx_scales,
                        F.n_cap, n_entries[f], r->ratio[f], cand, r->hsi_nb, r->hsi_blk, p->k,
                        topk, bmax, nullptr, ws + w.scores, w.blockmax - w.scores, stream,
                        stage_event(r, l, 2, 1), stage_event(r, l, 3, 0));
      if (st != CSA2_OK) return st;
      mark(r, l, 3, 1, stream);
      if (pool) {
        int32_t* c = L.cand_out ? L.cand_out : reinterpret_cast<int32_t*>(ws + w.cand);
        mark(r, l, 4, 0, stream);
        st = csa2_hsi_candidates(bmax, p->B, p->Tq, p->q_pos0, n_entries[l], r->ratio[l],
                                 r->hsi_blk, r->hsi_nb, c, stream);
        if (st != CSA2_OK) return st;
        mark(r, l, 4, 1, stream);
        slot_cand = c;
      }
      slot_topk = topk;
      slot_topk_layer = l;
    }
    // attention
    const void* kv = nullptr;
    const uint8_t *kv_codes = nullptr, *kv_scales = nullptr;
    const int32_t* topk = nullptr;
    int k = 0, n_cap = 0, n_ent = 0;
    if (md != CSA2_MODE_SWA) {
      const int f = r->kv_src[l];
      if (io[f].kv_codes) {
        kv_codes = io[f].kv_codes;
        kv_scales = io[f].kv_scales;
      } else {
        kv = io[f].kv_cache;
      }
      n_cap = io[f].n_cap;
      n_ent = n_entries[f];
      topk = slot_topk;
      k = p->k;
      if (slot_kv != f || !topk || slot_topk_layer != r->idx_src[l])
        return fail(CSA2_ERR_INVALID_ARG,
                    "layer %d: shared slots do not hold KV source %d / index source %d", l, f,
                    r->idx_src[l]);
    }
    mark(r, l, 5, 0, stream);
    st = csa2_sparse_attn_ex(L.q, p->B, p->Tq, p->H, p->q_pos0, kv, kv_codes, kv_scales, n_cap,
                             n_ent, topk, k, L.swa_codes ? nullptr : L.swa_kv, L.swa_codes,
                             L.swa_scales, L.swa_len, L.swa_pos0, p->window, L.sink, p->scale,
                             L.out, nullptr, ws + w.attn, w.total - w.attn, stream);
    if (st != CSA2_OK) return st;
    mark(r, l, 5, 1, stream);
  }
  return CSA2_OK;
}

}  // extern "C"
