// fp16 instantiation of the tcgen05 GEMM (hgemm_tcgen05.cuh) and the
// dispatcher's planning functions: tile width, block pairs, tail split.
#include "hgemm_tcgen05.cuh"

namespace gb300 {

int hgemm_pair_slots(int bn, int transA, int transB, int mode, int num_sms) {
  const bool A_MN = transA != 0, B_MN = transB == 0;
#define GB300_SLOTS(W, AM, BMN)                                                              \
  if (bn == W && A_MN == AM && B_MN == BMN)                                                  \
    return pair_slots<__half, W, AM, BMN, 2>(num_sms);
  GB300_SLOTS(128, false, true) GB300_SLOTS(128, true, true) GB300_SLOTS(128, false, false)
  GB300_SLOTS(128, true, false) GB300_SLOTS(256, false, true) GB300_SLOTS(256, true, true)
  GB300_SLOTS(256, false, false) GB300_SLOTS(256, true, false)
#undef GB300_SLOTS
  return num_sms / 2;
}

// Pairs of blocks share B tiles when the tile is 128 or 256 wide, there are at
// least two tile rows, and K is not split (the split-K path keeps single
// blocks).
bool hgemm_use_pair(int bn, int M, int splits, int allowed) {
  return allowed && (bn == 128 || bn == 256) && (M + BM - 1) / BM >= 2 && splits == 1;
}

// Tail split for the persistent grid (no split-K): with `workers` blocks (or
// pairs) taking units round-robin, the last round holds units % workers tiles.
// When that is at most half the workers, those tiles are cut into K slices so
// that the last round spreads over all workers.
TailPlan hgemm_plan_tail(int M, int N, int K, int bn, bool pair, int workers) {
  TailPlan t{0, 0, 0, 0, 0};
  const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + bn - 1) / bn;
  const int units = (pair ? (tiles_m + 1) / 2 : tiles_m) * tiles_n;
  const int full = units / workers, rem = units % workers;
  const int nkb = (K + BK - 1) / BK;
  if (workers <= 0 || full == 0 || rem == 0 || rem * 2 > workers || nkb < 8) return t;
  int sp = workers / rem;
  if (sp > nkb / 4) sp = nkb / 4;
  if (sp > 8) sp = 8;
  if (sp < 2) return t;
  const int per = (nkb + sp - 1) / sp;
  t.splits = (nkb + per - 1) / per;
  if (t.splits < 2) { t.splits = 0; return t; }
  t.k_slice = per * BK;
  t.dp_units = full * workers;
  const int halves = pair ? 2 : 1;
  t.ws_bytes = (size_t)rem * halves * t.splits * BM * bn * sizeof(float);
  // one counter per 32-row strip and epilogue column share (at most two)
  t.cnt_bytes = (size_t)rem * halves * 4 * 2 * sizeof(unsigned int);
  return t;
}

int hgemm_pick_bn(int M, int N, int transB, int num_sms, int batch) {
  // An MN-major B (transB == 0) is staged in 64-column swizzle atoms, so its
  // narrowest tile is 64 columns; a K-major B can go down to 32.
  if (N <= 32 && transB) return 32;
  if (N <= 64) return 64;
  if (N <= 128) return 128;
  // Wider N: the persistent grid runs ceil(tiles / SMs) rounds of tiles.  A
  // round of 128 x BN tiles costs, relative to BN = 256 and measured on GB300
  // at 4096^3 with 2-SM pairs: 0.85 (BN 128), 0.92 (BN 192), 1.0 (BN 256) --
  // narrower tiles re-read A more often per flop.  Pick the cheapest; ties go
  // to the wider tile.
  // (a strided batch multiplies the tile count: its entries share the rounds)
  const int64_t tm = (int64_t)((M + BM - 1) / BM) * (batch > 1 ? batch : 1);
  const int widths[3] = {256, 192, 128};
  const double round_cost[3] = {1.0, 0.92, 0.85};
  int best = 256;
  double best_cost = -1.0;
  for (int w = 0; w < 3; ++w) {
    const int64_t tiles = tm * ((N + widths[w] - 1) / widths[w]);
    const int64_t rounds = (tiles + num_sms - 1) / num_sms;
    const double cost = (double)rounds * round_cost[w];
    if (best_cost < 0.0 || cost < best_cost - 1e-9) { best = widths[w]; best_cost = cost; }
  }
  return best;
}

cudaError_t launch_hgemm(const HgemmArgs& a, LaunchCtx& ctx) {
  if (a.dtype == 2) return launch_hgemm_bf16(a, ctx);
  if (a.dtype == 3) return launch_hgemm_tf32(a, ctx);
  return launch_hgemm_t<__half>(a, ctx);
}

}  // namespace gb300
