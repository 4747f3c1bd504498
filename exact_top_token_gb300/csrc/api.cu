// api.cu -- the C ABI of the library (include/hytopk.h): argument checks,
// workspace layout and the launch sequence. Nothing here synchronises the
// stream or allocates memory.
#include <cstdint>
#include <cstring>

#include "launch.h"

using namespace hytopk;

namespace {

constexpr int kVersion = 100;  // 0.1.0

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool supported_h(int H) { return H >= 1 && H <= 128 && (H & (H - 1)) == 0; }
// key rows of 64, 128 or 256 bytes: bf16 keys d = 32, 64, 128; e4m3 keys d = 64, 128, 256
bool supported_d(int d, hytopk_dtype dt) {
  return dt != HYTOPK_E4M3 ? (d == 32 || d == 64 || d == 128) : (d == 64 || d == 128 || d == 256);
}
// bytes of a key element (also of the packed query operand, which takes the key type)
int elem_size(hytopk_dtype dt) { return dt == HYTOPK_E4M3 ? 1 : 2; }
bool valid_dtype(hytopk_dtype dt) {
  return dt == HYTOPK_BF16 || dt == HYTOPK_E4M3 || dt == HYTOPK_E4M3_BF16;
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int pad_queries(int n) { return (n + kQueryPad - 1) / kQueryPad * kQueryPad; }

struct SelectLayout {
  size_t perm, qpos, wq, qp, thr, cnt, cand, flist, failed, ctr, rowbuf, plan, total;
};

SelectLayout select_layout(int n, int L, int H, int d, int C, hytopk_dtype dt) {
  const size_t np = (size_t)pad_queries(n);
  SelectLayout s{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 1024);
    return at;
  };
  s.ctr = take(kCtrCount * sizeof(uint32_t));
  s.perm = take(np * 4);
  s.qpos = take(np * 4);
  s.thr = take(np * 4);
  s.cnt = take(np * 4);
  s.flist = take(np * 4);
  s.failed = take(np);
  s.wq = take(np * H * 4);
  s.qp = take(np * H * d * elem_size(dt));
  s.cand = take(np * (size_t)C * 8);
  s.rowbuf = take((size_t)kRecoveryCtas * L * 4);
  s.plan = take(((size_t)stream_chunks(L) + 1) * 4);
  s.total = off;
  return s;
}

int default_capacity(int k_top, int capacity) { return capacity > 0 ? capacity : 8 * k_top; }

// Rows per score-table chunk of the fallback past HYTOPK_MAX_RECOVERY_ROWS
// failed queries: whole rows of L scores in the candidate and recovery-row
// buffers (unused by then), in whole read-back waves (kTableCtas rows, one
// per CTA) when that takes no more chunks (a chunk a few rows past a wave
// leaves those rows to a second pass of the CTAs that took them).
int fallback_chunk_rows(const SelectLayout& lay, int n, int L) {
  size_t rows_fit = (lay.plan - lay.cand) / ((size_t)L * 4);
  if (rows_fit > (size_t)kTableCtas) {
    const size_t waves = rows_fit - rows_fit % kTableCtas;
    if ((n + waves - 1) / waves == (n + rows_fit - 1) / rows_fit) rows_fit = waves;
  }
  return (int)(rows_fit < (size_t)n ? rows_fit : (size_t)n);
}

Problem make_problem(const void* q, const float* q_scale, const void* k, const float* k_scale,
                     const float* w, const int32_t* positions, int n, int L, int H, int d,
                     int k_top, hytopk_dtype dt) {
  Problem p;
  p.q = q;
  p.q_scale = q_scale;
  p.k = k;
  p.k_scale = k_scale;
  p.w = w;
  p.positions = positions;
  p.n = n;
  p.L = L;
  p.H = H;
  p.d = d;
  p.k_top = k_top;
  p.dt = dt == HYTOPK_E4M3 ? 1 : 0;
  p.qdt = dt == HYTOPK_BF16 ? 0 : 1;
  return p;
}

#define HYTOPK_TRY(expr)                          \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return HYTOPK_CUDA_ERROR; \
  } while (0)

hytopk_status record(const hytopk_select_options* opts, int phase, cudaStream_t st) {
  if (opts && opts->phase_events && opts->phase_events[phase])
    if (cudaEventRecord(opts->phase_events[phase], st) != cudaSuccess) return HYTOPK_CUDA_ERROR;
  return HYTOPK_OK;
}

}  // namespace

namespace hytopk {

// Shape checks shared by every entry point.
hytopk_status check_shape(int n, int L, int H, int d, int k_top, hytopk_dtype dt) {
  if (n < 0 || L < 1 || H < 1 || d < 1 || k_top < 1 || !valid_dtype(dt)) return HYTOPK_INVALID_ARG;
  if (!supported_h(H) || !supported_d(d, dt) || k_top > kMaxTopK) return HYTOPK_UNSUPPORTED;
  if (n > (1 << 22) || L > (1 << 30)) return HYTOPK_UNSUPPORTED;
  return HYTOPK_OK;
}

hytopk_status check_inputs(const void* q, const float* q_scale, const void* k, const float* k_scale,
                           const float* w, hytopk_dtype dt, int n) {
  if (!k) return HYTOPK_INVALID_ARG;
  if (n > 0 && (!q || !w)) return HYTOPK_INVALID_ARG;
  // e4m3 rows carry a scale, bf16 rows none
  const bool q_e4m3 = dt != HYTOPK_BF16, k_e4m3 = dt == HYTOPK_E4M3;
  if (q_e4m3 ? (n > 0 && !q_scale) : (q_scale != nullptr)) return HYTOPK_INVALID_ARG;
  if (k_e4m3 ? !k_scale : (k_scale != nullptr)) return HYTOPK_INVALID_ARG;
  // rows are read in 16-byte pieces; scales and weights one fp32 at a time
  if ((q && !aligned16(q)) || !aligned16(k)) return HYTOPK_MISALIGNED;
  const float* fptrs[] = {q_scale, k_scale, w};
  for (const float* p : fptrs)
    if (p && (reinterpret_cast<uintptr_t>(p) & 3u) != 0) return HYTOPK_MISALIGNED;
  return HYTOPK_OK;
}

}  // namespace hytopk

extern "C" {

size_t hytopk_select_workspace_size(int n, int L, int H, int d, int k_top, int capacity,
                                    hytopk_dtype dt) {
  if (check_shape(n, L, H, d, k_top, dt) != HYTOPK_OK) return 0;
  const int C = default_capacity(k_top, capacity);
  if (capacity < 0 || C < k_top) return 0;
  return select_layout(n, L, H, d, C, dt).total;
}

int32_t hytopk_select_fallback_chunks(int n, int L, int H, int d, int k_top, int capacity,
                                      hytopk_dtype dt) {
  if (check_shape(n, L, H, d, k_top, dt) != HYTOPK_OK) return -1;
  const int C = default_capacity(k_top, capacity);
  if (capacity < 0 || C < k_top) return -1;
  if (n == 0) return 0;
  const int rows = fallback_chunk_rows(select_layout(n, L, H, d, C, dt), n, L);
  return rows > 0 ? (n + rows - 1) / rows : 0;
}

hytopk_status hytopk_select_ex(const void* q, const float* q_scale, const void* k,
                               const float* k_scale, const float* w, const int32_t* positions,
                               int n, int L, int H, int d, int k_top, hytopk_dtype dt,
                               int32_t* idx_out, float* scores_out, int capacity,
                               void* workspace, size_t workspace_bytes, hytopk_stats* stats_out,
                               const hytopk_select_options* opts, cudaStream_t stream) {
  hytopk_status s = check_shape(n, L, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  s = check_inputs(q, q_scale, k, k_scale, w, dt, n);
  if (s != HYTOPK_OK) return s;
  const int C = default_capacity(k_top, capacity);
  if (capacity < 0 || C < k_top) return HYTOPK_INVALID_ARG;
  if (n > 0 && (!positions || !idx_out || !workspace)) return HYTOPK_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return HYTOPK_MISALIGNED;
  const SelectLayout lay = select_layout(n, L, H, d, C, dt);
  if (workspace_bytes < lay.total) return HYTOPK_WORKSPACE_TOO_SMALL;
  if (n == 0) {
    if (stats_out) HYTOPK_TRY(cudaMemsetAsync(stats_out, 0, sizeof(hytopk_stats), stream));
    return HYTOPK_OK;
  }
  uint8_t* base = static_cast<uint8_t*>(workspace);
  SelectWs ws;
  ws.perm = reinterpret_cast<int32_t*>(base + lay.perm);
  ws.qpos = reinterpret_cast<int32_t*>(base + lay.qpos);
  ws.wq = reinterpret_cast<float*>(base + lay.wq);
  ws.qp = base + lay.qp;
  ws.thr = reinterpret_cast<float*>(base + lay.thr);
  ws.cnt = reinterpret_cast<int32_t*>(base + lay.cnt);
  ws.cand = reinterpret_cast<uint64_t*>(base + lay.cand);
  ws.failed_list = reinterpret_cast<int32_t*>(base + lay.flist);
  ws.failed = base + lay.failed;
  ws.counters = reinterpret_cast<uint32_t*>(base + lay.ctr);
  ws.rowbuf = reinterpret_cast<float*>(base + lay.rowbuf);
  ws.plan = reinterpret_cast<int32_t*>(base + lay.plan);
  ws.n_pad = pad_queries(n);
  ws.C = C;
  const Problem p = make_problem(q, q_scale, k, k_scale, w, positions, n, L, H, d, k_top, dt);
  const float* override_thr = opts ? opts->threshold_override : nullptr;
  const int reverse = opts ? opts->reverse_schedule : 0;

  if ((s = record(opts, HYTOPK_PHASE_PREP, stream)) != HYTOPK_OK) return s;
  HYTOPK_TRY(cudaMemsetAsync(ws.counters, 0, kCtrCount * sizeof(uint32_t), stream));
  HYTOPK_TRY(cudaMemsetAsync(ws.cnt, 0, (size_t)ws.n_pad * 4, stream));
  HYTOPK_TRY(launch_prep(p, ws, stream));
  if ((s = record(opts, HYTOPK_PHASE_THRESHOLD, stream)) != HYTOPK_OK) return s;
  HYTOPK_TRY(launch_threshold(p, ws, override_thr, stream));
  if ((s = record(opts, HYTOPK_PHASE_FILTER, stream)) != HYTOPK_OK) return s;
  HYTOPK_TRY(launch_filter(p, ws, reverse, stream));
  if ((s = record(opts, HYTOPK_PHASE_CHECK, stream)) != HYTOPK_OK) return s;
  HYTOPK_TRY(launch_check(p, ws, stream));
  if ((s = record(opts, HYTOPK_PHASE_SELECT, stream)) != HYTOPK_OK) return s;
  HYTOPK_TRY(launch_select(p, ws, idx_out, scores_out, stream));
  if ((s = record(opts, HYTOPK_PHASE_RECOVER, stream)) != HYTOPK_OK) return s;
  HYTOPK_TRY(launch_recover(p, ws, idx_out, scores_out, stream));
  {
    // Past HYTOPK_MAX_RECOVERY_ROWS failed queries every query is rescored
    // over its whole context: score-table rows in slot order, written into
    // the candidate and recovery-row buffers (unused by then) and read back
    // chunk by chunk. Whether that happens is known only on the device, so
    // these launches are always made and return at once without a fallback.
    float* table = reinterpret_cast<float*>(base + lay.cand);
    const int chunk = fallback_chunk_rows(lay, n, L);
    FallbackMaps maps;
    HYTOPK_TRY(prepare_fallback_table(p, ws, &maps));
    for (int slot0 = 0; chunk > 0 && slot0 < n; slot0 += chunk) {
      const int rows = n - slot0 < chunk ? n - slot0 : chunk;
      HYTOPK_TRY(launch_fallback_table(p, ws, maps, slot0, rows, table, stream));
      HYTOPK_TRY(launch_fallback_topk(p, ws, slot0, rows, table, idx_out, scores_out, stream));
    }
  }
  if ((s = record(opts, HYTOPK_NUM_PHASES, stream)) != HYTOPK_OK) return s;
  if (stats_out) HYTOPK_TRY(launch_finalize(ws, n, stats_out, stream));
  return HYTOPK_OK;
}

hytopk_status hytopk_select(const void* q, const float* q_scale, const void* k,
                            const float* k_scale, const float* w, const int32_t* positions, int n,
                            int L, int H, int d, int k_top, hytopk_dtype dt, int32_t* idx_out,
                            float* scores_out, int capacity, void* workspace,
                            size_t workspace_bytes, hytopk_stats* stats_out, cudaStream_t stream) {
  return hytopk_select_ex(q, q_scale, k, k_scale, w, positions, n, L, H, d, k_top, dt, idx_out,
                          scores_out, capacity, workspace, workspace_bytes, stats_out, nullptr,
                          stream);
}

hytopk_status hytopk_replay(const void* q, const float* q_scale, const void* k,
                            const float* k_scale, const float* w, const int32_t* idx, int n,
                            int L, int H, int d, int k_top, hytopk_dtype dt, float* scores_out,
                            uint32_t* dev_status, cudaStream_t stream) {
  hytopk_status s = check_shape(n, L, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  s = check_inputs(q, q_scale, k, k_scale, w, dt, n);
  if (s != HYTOPK_OK) return s;
  if (n == 0) return HYTOPK_OK;
  if (!idx || !scores_out) return HYTOPK_INVALID_ARG;
  const Problem p = make_problem(q, q_scale, k, k_scale, w, nullptr, n, L, H, d, k_top, dt);
  HYTOPK_TRY(launch_replay(p, idx, scores_out, dev_status, stream));
  return HYTOPK_OK;
}

hytopk_status hytopk_replay_grouped(const void* q, const float* q_scale, const void* k,
                                    const float* k_scale, const float* w, const int32_t* idx,
                                    int n, int L, int H, int d, int k_top, hytopk_dtype dt,
                                    int group, float* scores_out, uint32_t* dev_status,
                                    cudaStream_t stream) {
  if (group != 1 && group != 2) return HYTOPK_INVALID_ARG;
  hytopk_status s = check_shape(n, L, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  s = check_inputs(q, q_scale, k, k_scale, w, dt, n);
  if (s != HYTOPK_OK) return s;
  if (n == 0) return HYTOPK_OK;
  if (!idx || !scores_out) return HYTOPK_INVALID_ARG;
  const Problem p = make_problem(q, q_scale, k, k_scale, w, nullptr, n, L, H, d, k_top, dt);
  if (group == 2 && replay_pair_supported(p))
    HYTOPK_TRY(launch_replay_pair(p, idx, scores_out, dev_status, stream));
  else
    HYTOPK_TRY(launch_replay(p, idx, scores_out, dev_status, stream));
  return HYTOPK_OK;
}

// Two-pass workspace: the halved folded weights of the queries (padded by one
// query block), the bf16 copy of e4m3 queries for the mixed type, then the
// score-table chunk.
static size_t twopass_weights_bytes(int n, int H) {
  return align_up(((size_t)n + kQueryPad) * H * 4, 1024);
}
// e4m3 q against bf16 k: the table kernel reads q through a tensor map in the
// key element type, so q is first converted to a bf16 copy [n, H, d]
static size_t twopass_qconv_bytes(int n, int H, int d, hytopk_dtype dt) {
  return dt == HYTOPK_E4M3_BF16 ? align_up((size_t)n * H * d * 2, 1024) : 0;
}
static size_t twopass_fixed_bytes(int n, int L, int H, int d, hytopk_dtype dt) {
  return twopass_weights_bytes(n, H) + twopass_qconv_bytes(n, H, d, dt);
}

size_t hytopk_twopass_workspace_size(int n, int L, int H, int d, int k_top, hytopk_dtype dt,
                                     int rows_per_chunk) {
  if (check_shape(n, L, H, d, k_top, dt) != HYTOPK_OK) return 0;
  const int rows = rows_per_chunk <= 0 ? (n > 0 ? n : 1) : rows_per_chunk;
  return twopass_fixed_bytes(n, L, H, d, dt) + align_up((size_t)rows * L * 4, 1024);
}

hytopk_status hytopk_select_twopass(const void* q, const float* q_scale, const void* k,
                                    const float* k_scale, const float* w,
                                    const int32_t* positions, int n, int L, int H, int d,
                                    int k_top, hytopk_dtype dt, int32_t* idx_out,
                                    float* scores_out, void* workspace, size_t workspace_bytes,
                                    uint32_t* dev_status, cudaStream_t stream) {
  hytopk_status s = check_shape(n, L, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  s = check_inputs(q, q_scale, k, k_scale, w, dt, n);
  if (s != HYTOPK_OK) return s;
  if (n == 0) return HYTOPK_OK;
  if (!positions || !idx_out || !workspace) return HYTOPK_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return HYTOPK_MISALIGNED;
  const size_t fixed = twopass_fixed_bytes(n, L, H, d, dt);
  const size_t row_bytes = (size_t)L * 4;
  if (workspace_bytes < fixed + row_bytes) return HYTOPK_WORKSPACE_TOO_SMALL;
  size_t chunk = (workspace_bytes - fixed) / row_bytes;
  if (chunk > (size_t)n) chunk = (size_t)n;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  float* hw = reinterpret_cast<float*>(base);
  float* table = reinterpret_cast<float*>(base + fixed);
  const Problem p0 = make_problem(q, q_scale, k, k_scale, w, positions, n, L, H, d, k_top, dt);
  HYTOPK_TRY(launch_fold_weights(p0, n + kQueryPad, hw, stream));  // folds q_scale
  Problem p = p0;
  if (dt == HYTOPK_E4M3_BF16) {
    void* qconv = base + twopass_weights_bytes(n, H);
    HYTOPK_TRY(launch_convert_queries(p0, qconv, stream));
    p.q = qconv;
    p.qdt = 0;
  }
  for (int row0 = 0; row0 < n; row0 += (int)chunk) {
    const int rows = (int)((size_t)(n - row0) < chunk ? (size_t)(n - row0) : chunk);
    HYTOPK_TRY(launch_table(p, row0, rows, table, hw, dev_status, stream));
    HYTOPK_TRY(launch_table_topk(p, row0, rows, table, idx_out, scores_out, stream));
  }
  return HYTOPK_OK;
}

int32_t hytopk_sample_plan(int64_t ctx, int32_t k_top, int32_t* positions_out,
                           int32_t* rank_out) {
  if (ctx < 1 || k_top < 1) return 0;
  const int m = sample_count(ctx);
  if (positions_out)
    for (int j = 0; j < m; ++j) positions_out[j] = sample_position(ctx, m, j);
  if (rank_out) *rank_out = threshold_rank(ctx, k_top, m);
  return m;
}

const char* hytopk_status_string(hytopk_status status) {
  switch (status) {
    case HYTOPK_OK: return "ok";
    case HYTOPK_INVALID_ARG: return "invalid argument";
    case HYTOPK_UNSUPPORTED: return "unsupported shape or dtype";
    case HYTOPK_WORKSPACE_TOO_SMALL: return "workspace too small";
    case HYTOPK_CUDA_ERROR: return "CUDA error";
    case HYTOPK_MISALIGNED: return "device pointer misaligned";
  }
  return "unknown status";
}

int hytopk_version(void) { return kVersion; }

}  // extern "C"
