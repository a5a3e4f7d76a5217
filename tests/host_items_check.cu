// Host-side check of the prefill kernel's work decomposition (fa_items.cuh), built by
// tests/test_items_host.py with nvcc and run on the CPU.  For many problem shapes it walks every
// CTA's item list exactly as the kernel's roles do and checks:
//   1. every output row of every (sequence, query head) belongs to exactly one Q tile of one item;
//   2. an active tile's K/V range lies inside its item's union walk [u0, u1), so the softmax warps
//      of tile X and the MMA issuer make the same number of P handoffs (the named-barrier count
//      argument), and both equal handoffs_total_of;
//   3. the tile range covers every key any of its rows may see, and a tile the kernel leaves
//      unmasked holds only keys every valid row of the tile may see.
// Exit status 0 and "ok" when every check holds.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "fa_items.cuh"

using namespace fa;

static constexpr int BM = 128, BN = 128, NQT = 2;
static int g_fail = 0, g_cases = 0;

#define CHECK(cond, ...)                         \
  do {                                           \
    if (!(cond)) {                               \
      if (g_fail < 20) {                         \
        std::printf("FAIL %s: ", name);          \
        std::printf(__VA_ARGS__);                \
        std::printf("\n");                       \
      }                                          \
      ++g_fail;                                  \
    }                                            \
  } while (0)

// The launcher's choices: head pairs for an even group, rows per item, grid size.
static void run_case(const char* name, PrefillParams p, int max_rows, int sm_count) {
  ++g_cases;
  p.pair_heads = (p.group % 2 == 0) ? 1 : 0;
  const int rows_per_item = p.pair_heads ? BM : NQT * BM;
  p.n_qblk = (max_rows + rows_per_item - 1) / rows_per_item;
  const long long n_items_ll = (long long)(p.pair_heads ? p.Hq / 2 : p.Hq) * p.B * p.n_qblk;
  if (n_items_ll <= 0) return;
  const int n_items = (int)n_items_ll;
  const bool uniform = !p.cu_q && !p.seqlens_q && !p.seqlens_k;
  const long long G = uniform && n_items > sm_count ? sm_count : n_items;
  const int n_rounds = (int)((n_items + G - 1) / G);

  // rows_out and Lq per (sequence, head) from the geometry itself
  std::vector<int> seen;  // [b][h][row] coverage count
  std::vector<int> rows_out(p.B), base(p.B + 1, 0);
  for (int b = 0; b < p.B; ++b) {
    rows_out[b] = seq_info(p, b, 0).rows_out;
    base[b + 1] = base[b] + rows_out[b] * p.Hq;
  }
  seen.assign(base[p.B], 0);
  std::vector<int> item_seen(n_items, 0);

  for (long long c = 0; c < G; ++c) {
    uint32_t soft[2] = {0, 0}, issuer[2] = {0, 0};
    for (int k = 0; k < n_rounds; ++k) {
      const int w = snake_item_of(k, n_items, G, c);
      if (w < 0) continue;
      CHECK(w < n_items, "item %d out of range", w);
      item_seen[w]++;
      const WorkItem it = work_item<BM, BN>(p, w);
      if (!it.live) continue;
      for (int X = 0; X < NQT; ++X) {
        const QTileRange r = X ? it.rb : it.ra;
        const int h = item_head<BM>(p, it, X);
        const int q0 = item_row0<BM>(p, it, X);
        const int b = (w / (p.pair_heads ? p.Hq / 2 : p.Hq)) % p.B;
        CHECK(r.q0 == q0, "tile row %d vs %d", r.q0, q0);
        for (int i = q0; i < q0 + BM && i < it.s.rows_out; ++i) seen[base[b] + h * it.s.rows_out + i]++;
        if (r.t1 > r.t0) {
          soft[X] += (uint32_t)(r.t1 - r.t0);
          CHECK(it.u1 > it.u0 && r.t0 >= it.u0 && r.t1 <= it.u1, "tile range [%d,%d) outside [%d,%d)", r.t0, r.t1,
                it.u0, it.u1);
          // every visible key inside the range; unmasked tiles fully visible to every valid row
          for (int i = r.q0; i < r.q0 + BM && i < it.s.Lq; ++i) {
            int lo, hi;
            visible_keys(i + it.s.Lk - it.s.Lq, it.s.Lk, p.causal, p.window, lo, hi);
            if (hi > lo) CHECK(lo >= r.t0 * BN && hi <= r.t1 * BN, "row %d keys [%d,%d) outside tiles", i, lo, hi);
            for (int t = r.t0; t < r.t1; ++t)
              if (!tile_needs_mask<BN>(r, t * BN, it.s.Lk, p.causal, p.window))
                CHECK(lo <= t * BN && t * BN + BN <= hi, "tile %d left unmasked but row %d sees [%d,%d)", t, i, lo, hi);
          }
        }
      }
      if (it.u1 > it.u0)
        for (int t = it.u0; t < it.u1; ++t)
          for (int X = 0; X < NQT; ++X) {
            const QTileRange r = X ? it.rb : it.ra;
            if (t >= r.t0 && t < r.t1) issuer[X]++;
          }
    }
    for (int X = 0; X < NQT; ++X) {
      CHECK(soft[X] == issuer[X], "CTA %lld tile %d: softmax %u vs issuer %u handoffs", c, X, soft[X], issuer[X]);
      const uint32_t total = handoffs_total_of<BM, BN>(p, X, n_rounds, n_items, G, c);
      CHECK(soft[X] == total, "CTA %lld tile %d: handoffs_total %u vs %u", c, X, total, soft[X]);
    }
  }
  for (int w = 0; w < n_items; ++w) CHECK(item_seen[w] == 1, "item %d taken %d times", w, item_seen[w]);
  for (size_t e = 0; e < seen.size(); ++e) CHECK(seen[e] == 1, "output row %zu covered %d times", e, seen[e]);
}

static PrefillParams base_params(int B, int Hq, int Hkv, int Nq, int Nk, int causal, int window) {
  PrefillParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.group = Hq / Hkv;
  p.causal = causal;
  p.window = window;
  return p;
}

int main() {
  char name[160];
  const int heads[][2] = {{1, 1}, {2, 1}, {3, 3}, {4, 2}, {8, 8}, {12, 4}, {32, 8}};
  const int lens[] = {1, 100, 128, 129, 256, 300, 1024, 4096};
  const int windows[] = {0, 1, 17, 127, 128, 129, 300, 1024};
  const int sms[] = {152, 7};
  // dense, including Nq != Nk
  for (auto& hd : heads)
    for (int nq : lens)
      for (int nk : {nq, nq + 1, nq + 63, nq + 126, nq + 127, nq > 1 ? nq - 1 : 1, nq * 2 + 3, nq > 1 ? nq / 2 : 1})
        for (int causal = 0; causal < 2; ++causal)
          for (int win : windows)
            for (int sm : sms) {
              std::snprintf(name, sizeof name, "dense Hq=%d Hkv=%d Nq=%d Nk=%d causal=%d window=%d sms=%d", hd[0], hd[1],
                            nq, nk, causal, win, sm);
              run_case(name, base_params(2, hd[0], hd[1], nq, nk, causal, win), nq, sm);
            }
  // padded (per-sequence lengths, zeros included) and packed (cu_seqlens), seeded
  unsigned seed = 12345;
  auto rnd = [&](int n) {
    seed = seed * 1103515245u + 12345u;
    return (int)((seed >> 8) % (unsigned)n);
  };
  for (int rep = 0; rep < 400; ++rep) {
    const auto& hd = heads[rnd(7)];
    const int B = 1 + rnd(6), N = 1 + rnd(1200), causal = rnd(2), win = windows[rnd(8)];
    std::vector<int> lq(B), lk(B), cq(B + 1, 0), ck(B + 1, 0);
    int maxq = 0, maxk = 0;
    for (int b = 0; b < B; ++b) {
      lq[b] = rnd(5) == 0 ? 0 : 1 + rnd(N);
      lk[b] = causal ? lq[b] + rnd(300) : rnd(5) == 0 ? 0 : 1 + rnd(N);
      cq[b + 1] = cq[b] + lq[b];
      ck[b + 1] = ck[b] + lk[b];
      maxq = lq[b] > maxq ? lq[b] : maxq;
      maxk = lk[b] > maxk ? lk[b] : maxk;
    }
    PrefillParams pp = base_params(B, hd[0], hd[1], N, N + 300, causal, win);
    pp.seqlens_q = lq.data();
    pp.seqlens_k = lk.data();
    std::snprintf(name, sizeof name, "padded rep=%d B=%d Hq=%d N=%d causal=%d window=%d", rep, B, hd[0], N, causal, win);
    run_case(name, pp, N, 152);
    if (maxq == 0) continue;
    PrefillParams pk = base_params(B, hd[0], hd[1], maxq, maxk > 0 ? maxk : 1, causal, win);
    pk.cu_q = cq.data();
    pk.cu_k = ck.data();
    pk.total_q = cq[B];
    pk.total_k = ck[B];
    std::snprintf(name, sizeof name, "packed rep=%d B=%d Hq=%d maxq=%d causal=%d window=%d", rep, B, hd[0], maxq, causal,
                  win);
    run_case(name, pk, maxq, 152);
  }
  if (g_fail) {
    std::printf("%d failures in %d cases\n", g_fail, g_cases);
    return 1;
  }
  std::printf("ok %d cases\n", g_cases);
  return 0;
}
