// fp16 instantiation of the tcgen05 GEMM (hgemm_tcgen05.cuh) and the
// dispatcher's planning functions: tile width, block pairs, schedule.
#include "hgemm_tcgen05.cuh"

namespace gb300 {

int hgemm_pair_slots(int bn, int transA, int transB, int num_sms) {
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

// Pairs of blocks run 2-SM MMAs when the tile is 128 or 256 wide and there
// are at least two tile rows.
bool hgemm_use_pair(int bn, int M, int allowed) {
  return allowed == 2 && (bn == 128 || bn == 256) && (M + BM - 1) / BM >= 2;
}

// Fewest K steps a stream-K range gets; most ranges that share one tile; and
// what finishing shared tiles costs, in K steps of the busiest worker:
// publishing partial sums, and the last contributor reading them back and
// adding them before its store (compile-time knobs).  Measured on GB300 with
// fp16: for 2-SM pairs of 256-wide tiles, sharing that shortens the busiest
// worker by 14 K steps loses (512 x 5632 x 2048: 21 -> 33 us), by 40 gains
// nothing (4096^3), by 66 still loses a little (512 x 2048 x 5632: 35.5 ->
// 36.5 us) and by 96 gains (1024 x 1024 x 8192: 45.7 -> 39.6 us); single
// 64-wide tiles, whose partial sums are a quarter the size, gain from 24
// steps up (512 x 32 x 2048: 17.0 -> 16.1 us; 512 x 32 x 5632: 31.4 -> 22.3
// us).
#ifndef GB300_HG_SK_MIN_STEPS
#define GB300_HG_SK_MIN_STEPS 4
#endif
#ifndef GB300_HG_SK_MAX_CONTRIB
#define GB300_HG_SK_MAX_CONTRIB 5
#endif
#ifndef GB300_HG_SK_COST_WIDE
#define GB300_HG_SK_COST_WIDE 72
#endif
#ifndef GB300_HG_SK_COST_NARROW
#define GB300_HG_SK_COST_NARROW 16
#endif
// ... and when every contributor publishes and a reduction kernel finishes
// (wide tiles; 64-wide or narrower: 512 x 32 x 2048 fp16, 16 ranges of 8
// steps against 4 tiles of 32: 17.0 -> 15.0 us)
#ifndef GB300_HG_SK_COST_PUBLISH
#define GB300_HG_SK_COST_PUBLISH 24
#endif
#ifndef GB300_HG_SK_COST_PUBLISH_NARROW
#define GB300_HG_SK_COST_PUBLISH_NARROW 12
#endif
// Most ranges that share one tile of 64 columns or fewer when a reduction
// kernel finishes it (its threads load every contributor's partial sums at
// once): 512 x 32 x 5632 fp16, 16 ranges of 22 steps against 28 of 12.6:
// 14.9 -> 12.4 us.  Wider tiles keep GB300_HG_SK_MAX_CONTRIB: 512 x 2048 x
// 5632 on 2-SM pairs, 64 ranges of 22 steps (four to a tile, none straddling
// two) against 76 of 18.5: 24.7 against 30.9 us.
#ifndef GB300_HG_SK_MAX_CONTRIB_PUBLISH
#define GB300_HG_SK_MAX_CONTRIB_PUBLISH 16
#endif

// K steps a stream-K plan adds for finishing shared tiles (0 without).
int sk_cost_steps(const HPlan& pl) {
  if (pl.sk_workers == 0) return 0;
  if (pl.sk_publish)
    return pl.bn <= 64 ? GB300_HG_SK_COST_PUBLISH_NARROW : GB300_HG_SK_COST_PUBLISH;
  return pl.bn <= 64 ? GB300_HG_SK_COST_NARROW : GB300_HG_SK_COST_WIDE;
}

// K steps the busiest worker of a plan runs.
int64_t busiest_steps(const HPlan& pl) {
  int64_t s = (int64_t)((pl.dp_tiles + pl.workers - 1) / pl.workers) * pl.steps;
  if (pl.sk_workers > 0) s += (pl.sk_steps + pl.sk_workers - 1) / pl.sk_workers;
  return s;
}

HPlan hgemm_plan(int M, int N, int K, int bn, int transA, int transB, int kstep, int batch,
                 int pair_allowed, int num_sms, int sk_mode) {
  HPlan pl;
  pl.bn = bn;
  const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + bn - 1) / bn;
  const bool pair = hgemm_use_pair(bn, M, pair_allowed);
  pl.pair = pair ? 2 : 0;
  const int64_t rows = pair ? (tiles_m + 1) / 2 : tiles_m;
  const int64_t nb = batch > 1 ? batch : 1;
  const int64_t tiles = rows * tiles_n * nb;
  const int steps = (K + kstep - 1) / kstep;
  const int wmax = pair ? hgemm_pair_slots(bn, transA, transB, num_sms) : num_sms;
  pl.tiles = (int)tiles;
  pl.steps = steps > 0 ? steps : 1;
  pl.dp_tiles = (int)tiles;
  pl.workers = (int)(tiles < wmax ? tiles : wmax);
  if (sk_mode != 0 && nb == 1 && tiles > 0 && steps >= 2 * GB300_HG_SK_MIN_STEPS) {
    // Tiles of the last, part-filled round are shared, together with the
    // round before it when there is one: every range then spans at least a
    // tile, so a shared tile has two contributors -- one range's first unit
    // (early) and the previous range's last (late), which finds the other's
    // partial sums waiting.  Mode 2 shares every tile.
    const int64_t rem = tiles % wmax;
    int64_t shared = rem == 0 ? 0 : (tiles >= 2 * (int64_t)wmax ? rem + wmax : tiles);
    if (sk_mode >= 2) shared = tiles;
    // With every tile shared, all ranges end together and race to finish
    // their tiles; there a reduction kernel over the published sums (every
    // SM taking part) beats the last contributor's finish (one block or block
    // pair a tile).
    const int64_t total = shared * steps;
    const bool publish = sk_mode == 3 || (sk_mode == 1 && tiles == shared);
    int64_t skw = total / GB300_HG_SK_MIN_STEPS;
    if (skw > wmax) skw = wmax;
    // at most GB300_HG_SK_MAX_CONTRIB(_PUBLISH) ranges meet in a tile
    const int64_t cap = shared * ((publish && bn <= 64 ? GB300_HG_SK_MAX_CONTRIB_PUBLISH
                                                       : GB300_HG_SK_MAX_CONTRIB) - 1);
    if (skw > cap) skw = cap;
    // (positions up to skw * total must fit 64 bits; every range non-empty)
    if (shared > 0 && skw >= 2 && total < ((int64_t)1 << 40)) {
      HPlan sk = pl;
      sk.dp_tiles = (int)(tiles - shared);
      sk.sk_workers = (int)skw;
      sk.sk_steps = total;
      sk.workers = sk.dp_tiles > 0 ? wmax : (int)skw;
      const int P = pair ? 2 : 1;
      sk.ws_bytes = (size_t)skw * 2 * P * BM * bn * sizeof(float);
      sk.sk_publish = publish;
      sk.cnt_bytes =
          sk.sk_publish ? 0 : (size_t)shared * P * 4 * EPI_HALVES * sizeof(unsigned int);
      // shared only where the busiest worker saves more than finishing the
      // shared tiles costs
      if (sk_mode >= 2 || busiest_steps(sk) + sk_cost_steps(sk) < busiest_steps(pl)) pl = sk;
    }
  }
  // Epilogue warps per accumulator quarter.  The epilogue of one unit is
  // bound by its warps' issue latency (about 1 us per 32 x 64 block a warp
  // stores, measured on GB300), which the next unit's main loop hides except
  // after a worker's last unit, where it adds to the launch: both shares of
  // warps drain it when units are short (<= GB300_HG_EPI2_STEPS K steps)
  // (4096 x 4096 x 128 fp16: 23.2 -> 19-21 us with both).
#ifndef GB300_HG_EPI2_STEPS
#define GB300_HG_EPI2_STEPS 8
#endif
  int64_t unit_steps = pl.steps;
  if (pl.sk_workers > 0) {
    const int64_t per = (pl.sk_steps + pl.sk_workers - 1) / pl.sk_workers;
    if (per < unit_steps) unit_steps = per;
  }
  // (a 32-wide tile is one 32-column chunk: nothing to share; with every
  // tile shared, every worker's epilogue is the publishing of its partial
  // sums at the end of the launch: both shares)
  pl.epi_halves = (EPI_HALVES > 1 && bn >= 64 &&
                   (unit_steps <= GB300_HG_EPI2_STEPS || pl.sk_publish)) ? EPI_HALVES : 1;
  return pl;
}

int hgemm_pick_bn(int M, int N, int K, int transA, int transB, int kstep, int batch,
                  int pair_allowed, int num_sms, int sk_mode) {
  // An MN-major B (transB == 0) is staged in 64-column swizzle atoms, so its
  // narrowest tile is 64 columns; a K-major B can go down to 32.
  if (N <= 32 && transB) return 32;
  if (N <= 64) return 64;
  if (N <= 128) return 128;
  // Wider N: the launch takes as long as its busiest worker, which runs
  // ceil(whole tiles / workers) tiles of `steps` K steps plus its stream-K
  // range (and the finishing of shared tiles).  A K step of a 128 x BN tile
  // costs, relative to BN = 256 and measured on GB300 at 4096^3 with 2-SM
  // pairs: 0.85 (BN 128), 0.92 (BN 192), 1.0 (BN 256) -- narrower tiles
  // re-read A more often per flop.  Pick the cheapest; ties go to the wider
  // tile.
  const int widths[3] = {256, 192, 128};
  const double step_cost[3] = {1.0, 0.92, 0.85};
  int best = 256;
  double best_cost = -1.0;
  for (int w = 0; w < 3; ++w) {
    const HPlan pl = hgemm_plan(M, N, K, widths[w], transA, transB, kstep, batch, pair_allowed,
                                num_sms, sk_mode);
    const double cost = (double)(busiest_steps(pl) + sk_cost_steps(pl)) * step_cost[w];
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
