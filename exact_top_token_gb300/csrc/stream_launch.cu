// stream_launch.cu -- host launchers of the streaming engine: the fused
// score + filter phase of hytopk_select and the table writer of the two-pass
// path.
#include "launch.h"
#include "stream_engine.cuh"

namespace hytopk {

cudaError_t launch_stream_d64_bf16(int H, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                                   const stream::Args& a, int grid, cudaStream_t st);
cudaError_t launch_stream_d64_e4m3(int H, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                                   const stream::Args& a, int grid, cudaStream_t st);
cudaError_t launch_stream_d128_bf16(int H, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                                    const stream::Args& a, int grid, cudaStream_t st);
cudaError_t launch_stream_d128_e4m3(int H, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                                    const stream::Args& a, int grid, cudaStream_t st);
cudaError_t launch_stream_d32_bf16(int H, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                                   const stream::Args& a, int grid, cudaStream_t st);
cudaError_t launch_stream_d256_e4m3(int H, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                                    const stream::Args& a, int grid, cudaStream_t st);

namespace {

int row_bytes(const Problem& p) { return p.d * (p.dt == 0 ? 2 : 1); }
int atom_bytes(const Problem& p) { return row_bytes(p) >= 128 ? 128 : 64; }

cudaError_t dispatch(const Problem& p, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                     const stream::Args& a, int grid, cudaStream_t st) {
  if (p.dt == 0) {
    if (p.d == 32) return launch_stream_d32_bf16(p.H, mode, km, qm, a, grid, st);
    if (p.d == 64) return launch_stream_d64_bf16(p.H, mode, km, qm, a, grid, st);
    return launch_stream_d128_bf16(p.H, mode, km, qm, a, grid, st);
  }
  if (p.d == 64) return launch_stream_d64_e4m3(p.H, mode, km, qm, a, grid, st);
  if (p.d == 128) return launch_stream_d128_e4m3(p.H, mode, km, qm, a, grid, st);
  return launch_stream_d256_e4m3(p.H, mode, km, qm, a, grid, st);
}

bool key_map(const Problem& p, CUtensorMap* km) {
  const int es = p.dt == 0 ? 2 : 1;
  return make_tmap_2d(km, p.k, p.dt, (uint64_t)p.d, (uint64_t)p.L, atom_bytes(p) / es, 128,
                      atom_bytes(p));
}

}  // namespace

// one MMA group of 256 (query, head) columns per work item
int stream_query_block(int H, int /*d*/, int /*dt*/) { return 256 / H; }

cudaError_t launch_filter(const Problem& p, const SelectWs& ws, int reverse, cudaStream_t st) {
  if (ws.n_pad == 0) return cudaSuccess;
  const int es = p.dt == 0 ? 2 : 1;
  CUtensorMap km, qm;
  if (!key_map(p, &km)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&qm, ws.qp, p.dt, (uint64_t)p.d, (uint64_t)ws.n_pad * p.H,
                    atom_bytes(p) / es, 256, atom_bytes(p)))
    return cudaErrorInvalidValue;
  const int qb = stream_query_block(p.H, p.d, p.dt);
  // The long key chunks (fewer item boundaries, each a reload of the block's
  // query operand and weights) when they still leave 64 work items per SM
  // before the causal cut, and when a query's expected candidates per item
  // (about 3k of its keys pass, spread over a context of up to L keys) fit
  // its staging room (past it, keys take one global atomic each).
  const int long_keys = stream::kChunkTilesLong * kTileKeys;
  const int64_t long_items = (int64_t)(ws.n_pad / qb) * ((p.L + long_keys - 1) / long_keys);
  const double per_item = 3.0 * p.k_top * (double)long_keys / (double)p.L;
  const bool long_chunks = long_items >= 64LL * num_sms() &&
                           per_item <= (double)stream::stage_capacity(p.H, qb);
  const int chunk_tiles = long_chunks ? stream::kChunkTilesLong : stream::kChunkTiles;
  cudaError_t e = launch_plan(ws, p.L, qb, chunk_tiles, st);
  if (e != cudaSuccess) return e;
  stream::Args a{};
  a.chunk_tiles = chunk_tiles;
  a.qpos = ws.qpos;
  a.thr = ws.thr;
  a.wq = ws.wq;
  a.cnt = ws.cnt;
  a.cand = ws.cand;
  a.plan = ws.plan;
  a.C = ws.C;
  a.n_pad = ws.n_pad;
  a.reverse = reverse;
  a.k_scale = p.k_scale;
  a.L = p.L;
  a.status = ws.counters + kCtrStatus;
  a.work = ws.counters + kCtrFilterWork;  // zeroed with the counters at the call's start
  return dispatch(p, 0, km, qm, a, num_sms(), st);
}

cudaError_t prepare_fallback_table(const Problem& p, const SelectWs& ws, FallbackMaps* m) {
  const int es = p.dt == 0 ? 2 : 1;
  if (!key_map(p, &m->km)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&m->qm, ws.qp, p.dt, (uint64_t)p.d, (uint64_t)ws.n_pad * p.H,
                    atom_bytes(p) / es, 256, atom_bytes(p)))
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

cudaError_t launch_fallback_table(const Problem& p, const SelectWs& ws, const FallbackMaps& m,
                                  int slot0, int rows, float* table, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const CUtensorMap& km = m.km;
  const CUtensorMap& qm = m.qm;
  stream::Args a{};
  a.chunk_tiles = stream::kChunkTiles;
  a.wq = ws.wq;  // halved folded weights in slot order
  a.positions = ws.qpos;
  a.table = table;
  a.row0 = slot0;
  a.rows = rows;
  a.n = ws.n_pad;
  a.k_scale = p.k_scale;
  a.L = p.L;
  a.status = ws.counters + kCtrStatus;
  a.gate = ws.counters + kCtrFailed;
  return dispatch(p, 1, km, qm, a, num_sms(), st);
}

cudaError_t launch_table(const Problem& p, int row0, int rows, float* table, const float* hw,
                         uint32_t* status, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int es = p.dt == 0 ? 2 : 1;
  CUtensorMap km, qm;
  if (!key_map(p, &km)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&qm, p.q, p.dt, (uint64_t)p.d, (uint64_t)p.n * p.H, atom_bytes(p) / es, 256,
                    atom_bytes(p)))
    return cudaErrorInvalidValue;
  stream::Args a{};
  // long key chunks when they still leave 64 work items per SM, as in the
  // filter (every score is written, so no staging bound)
  const int qb = stream_query_block(p.H, p.d, p.dt);
  const int long_keys = stream::kChunkTilesLong * kTileKeys;
  const int64_t long_items =
      (int64_t)((rows + qb - 1) / qb) * ((p.L + long_keys - 1) / long_keys);
  a.chunk_tiles = long_items >= 64LL * num_sms() ? stream::kChunkTilesLong : stream::kChunkTiles;
  a.wq = hw;
  a.w = p.w;
  a.q_scale = p.q_scale;
  a.positions = p.positions;
  a.table = table;
  a.row0 = row0;
  a.rows = rows;
  a.n = p.n;
  a.k_scale = p.k_scale;
  a.L = p.L;
  a.status = status;
  return dispatch(p, 1, km, qm, a, num_sms(), st);
}

}  // namespace hytopk
