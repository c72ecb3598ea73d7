// Host-side check of the split-KV work plan (kvq_make_plan + kvq_plan_cuts +
// plan_unit_chunks) over many random layouts: every unit's positions are
// covered exactly once by the chunks' pieces, the per-unit chunk ranges
// agree with a brute-force scan (and so does the most chunks of any unit),
// multi-query plans have their unit count, partial slots u + c are unique, visual cuts
// of packed units are 16-row aligned, and with at least as many chunks as
// units no chunk holds work of two units.  Cluster-mode plans (cs chunks per
// unit, unit u on chunks u * cs .. u * cs + cs - 1) are drawn too.  Prints
// "ok" or the first failure.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <set>
#include <vector>

#include "kvq_internal.h"

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static uint32_t next(uint32_t n) {
  rng ^= rng << 13;
  rng ^= rng >> 7;
  rng ^= rng << 17;
  return static_cast<uint32_t>(rng % n);
}

#define FAIL(...)                      \
  do {                                 \
    std::printf(__VA_ARGS__);          \
    std::printf("\n");                 \
    return 1;                          \
  } while (0)

// Staged-tile geometry for every bit-width and group size: at least one
// 32-row block per tile, whole multiples of 32 rows, and the sub-buffers
// (each a multiple of 128 bytes) inside one stage.
static int check_tiles() {
  const int bits[] = {2, 4, 8, 16};
  const int groups[] = {32, 64, 128};
  for (int kb : bits)
    for (int vb : bits)
      for (int G : groups) {
        const int krow = 16 * kb, vrow = 16 * vb;
        const int ksz = kb < 16 ? 4 * (kvq::kD / G) : 0, vsz = vb < 16 ? 4 * (kvq::kD / G) : 0;
        const int tt = kvq::packed_tile_rows32(krow + vrow + ksz + vsz);
        const int ttk = kvq::packed_tile_rows32(2 * kvq::kD + vrow + vsz);
        for (int t : {tt, ttk}) {
          if (t < 32 || t % 32) FAIL("tile of %d rows for K%d V%d G%d", t, kb, vb, G);
        }
        if (tt * (krow + vrow + ksz + vsz) > kvq::kStageBytes) FAIL("packed tile overflows (K%d V%d G%d)", kb, vb, G);
        if ((tt * krow) % 128 || (tt * vrow) % 128 || (tt * ksz) % 128)
          FAIL("sub-buffer not 128-byte aligned (K%d V%d G%d)", kb, vb, G);
        if (ttk * (2 * kvq::kD + vrow + vsz) > kvq::kStageBytes) FAIL("K-only tile overflows (V%d G%d)", vb, G);
      }
  return 0;
}

int main(int argc, char** argv) {
  const int cases = argc > 1 ? std::atoi(argv[1]) : 3000;
  if (check_tiles()) return 1;
  static kvq::Cut cuts[KVQ_MAX_CTAS + 1];
  int n_aligned = 0, n_stream = 0, n_cluster = 0;
  for (int it = 0; it < cases; ++it) {
    kvq_layout_desc d;
    std::memset(&d, 0, sizeof(d));
    const int bs[] = {1, 2, 3, 8, 16, 32};
    const int hs[] = {1, 2, 4, 8, 32, 40};
    const int gs[] = {1, 2, 7, 8, 9, 16};
    const int bits[] = {2, 4, 8, 16};
    const int groups[] = {32, 64, 128};
    d.B = bs[next(6)];
    d.H_kv = hs[next(6)];
    d.H_q = d.H_kv * gs[next(6)];
    if (d.H_q > KVQ_MAX_HEADS) d.H_q = d.H_kv;
    d.D = 128;
    d.T_cap = 1 + static_cast<int>(next(40000));
    d.vis_start = static_cast<int>(next(static_cast<uint32_t>(d.T_cap) + 1));
    d.vis_end = d.vis_start + static_cast<int>(next(static_cast<uint32_t>(d.T_cap - d.vis_start) + 1));
    d.k_bits = bits[next(4)];
    d.v_bits = bits[next(4)];
    d.group_size = groups[next(3)];
    for (int h = 0; h < d.H_kv; ++h) {
      const uint32_t r = next(8);
      d.protected_heads[h] = r == 0 ? 1 : (r == 1 ? 2 : 0);  // some protected, some K-only
    }
    kvq_layout L;
    if (kvq_cache_layout(&d, &L) != KVQ_OK) FAIL("layout rejected at case %d", it);
    const int T = 1 + static_cast<int>(next(static_cast<uint32_t>(d.T_cap)));
    const int targets[] = {1, 7, 152, 304, 1024};
    const int nqs[] = {1, 1, 2, 3, 8, 64};  // query tokens (multi-query plans have more units)
    const int n_q = nqs[next(6)];
    kvq::Plan P = kvq_make_plan(&L, T, targets[next(5)], n_q);
    if (P.U != d.B * d.H_kv * ((L.g * n_q + kvq::kNH - 1) / kvq::kNH)) FAIL("case %d: unit count", it);
    const int css[] = {2, 4, 8, 16};
    const int cs = css[next(4)];
    const bool cluster_mode = next(3) == 0 && P.U * cs <= KVQ_MAX_CTAS;
    if (cluster_mode) P.cs = cs;
    kvq_plan_cuts(&P, cuts);
    (cluster_mode ? n_cluster : (P.aligned ? n_aligned : n_stream))++;
    if (cluster_mode && (P.C != P.U * cs || !P.aligned)) FAIL("case %d: cluster plan has %d chunks", it, P.C);
    if (cuts[0].u != 0 || cuts[0].p != 0) FAIL("case %d: cut 0 = (%d,%d)", it, cuts[0].u, cuts[0].p);
    if (cuts[P.C].u != P.U || cuts[P.C].p != 0) FAIL("case %d: last cut", it);
    std::vector<int> covered(P.U, 0);  // next uncovered position of each unit
    std::set<long> slots;
    for (int c = 0; c < P.C; ++c) {
      const kvq::Cut a = cuts[c], e = cuts[c + 1];
      if (e.u < a.u || (e.u == a.u && e.p < a.p)) FAIL("case %d: cuts not monotone at %d", it, c);
      const int ul = kvq::chunk_last_unit(cuts, c, P.U);
      int work_units = 0;
      for (int u = a.u; u <= ul; ++u) {
        const int ps = u == a.u ? a.p : 0;
        const int pe = u == e.u ? e.p : P.T;
        if (ps != covered[u]) FAIL("case %d: unit %d piece starts at %d, expected %d", it, u, ps, covered[u]);
        if (pe < ps) FAIL("case %d: negative piece", it);
        covered[u] = pe;
        if (pe > ps) ++work_units;
        if (!slots.insert(static_cast<long>(u) + c).second) FAIL("case %d: slot %d reused", it, u + c);
        const bool bf16_only = kvq::unit_class(P, u) == kvq::kClsProt;
        if (!bf16_only && ps > P.vsa && ps < P.vea && (ps - P.vsa) % kvq::kVisAlign)
          FAIL("case %d: unaligned visual cut %d", it, ps);
      }
      if (P.aligned && work_units > 1) FAIL("case %d: chunk %d spans %d units", it, c, work_units);
    }
    int most = 0;
    for (int u = 0; u < P.U; ++u) {
      if (covered[u] != P.T) FAIL("case %d: unit %d covered to %d of %d", it, u, covered[u], P.T);
      int bf = -1, bl = -1;
      for (int c = 0; c < P.C; ++c)
        if (cuts[c].u <= u && kvq::chunk_last_unit(cuts, c, P.U) >= u) {
          if (bf < 0) bf = c;
          if (bl >= 0 && c != bl + 1) FAIL("case %d: unit %d chunks not contiguous", it, u);
          bl = c;
        }
      int cf, cl;
      kvq::plan_unit_chunks(P, cuts, u, &cf, &cl);
      if (cluster_mode && (cf != u * cs || cl != u * cs + cs - 1))
        FAIL("case %d: cluster unit %d on chunks [%d,%d]", it, u, cf, cl);
      if (cf != bf || cl != bl)
        FAIL("case %d (aligned %d): unit %d chunks [%d,%d], brute force [%d,%d]", it, P.aligned, u, cf, cl, bf, bl);
      if (bl - bf + 1 > most) most = bl - bf + 1;
    }
    if (kvq::plan_max_unit_chunks(P, cuts) != most)
      FAIL("case %d (aligned %d): most chunks per unit %d, brute force %d", it, P.aligned,
           kvq::plan_max_unit_chunks(P, cuts), most);
  }
  std::printf("ok %d cases (%d per-unit, %d stream, %d cluster)\n", cases, n_aligned, n_stream, n_cluster);
  return 0;
}
