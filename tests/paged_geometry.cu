#include <cstdio>
#include <cstdlib>
// Host enumeration of the paged cache's tile geometry (kvq_internal.h:
// paged_tiles, paged_tile, for_each_paged_copy) over every consistent
// per-sequence state of several shapes, with the general kernel's tile sizes
// and (d_h 128, G >= 32) the tensor-core kernel's: tiles cover [0, L) in
// order, fit a stage, never cross a page, and every bulk copy is 16-byte
// aligned, inside its page or ring, and adds up to the tile's expected byte
// count; for the tensor-core kernel also at most kTcMaxGroups K groups a
// tile and 32-token units inside one K group.  Built and
// run on the CPU by tests/test_paged_cpu.py; exits nonzero on a bad tile.
#include "../quantized_kv_cache_kivi_gb300/csrc/kvq_internal.h"
using namespace kvq;
static int stage_bytes(int t, int kb, int vb, int d, int G, int Gv) {
  auto a16 = [](int x) { return (x + 15) & ~15; };
  int b = a16(t * d * kb / 8) + a16(t * d * vb / 8);
  if (kb != 16) b += 2 * ((t + G - 1) / G + 1) * d * 2;
  if (vb != 16) b += 2 * a16(t * (d / Gv) * 2);
  return b;
}
static bool fits(int t, int kb, int vb, int d, int G, int Gv, int gq) {
  if (stage_bytes(t, kb, vb, d, G, Gv) > kStageBytes) return false;
  return kb == 16 || ((t + G - 1) / G + 1) * gq * d * 4 <= kQsBytes;
}
static bool tc_fits(int t, int kb, int vb, int d, int G, int Gv) {
  return stage_bytes(t, kb, vb, d, G, Gv) <= kTcStageBytes && (kb == 16 || (t + G - 1) / G + 1 <= kTcMaxGroups);
}
int main() {
  long long checked = 0, bad = 0;
  int cfgs[][8] = {  // d, G, Gv, R, bits, P, maxp, gq
    {128, 32, 32, 64, 2, 128, 7, 1}, {128, 32, 32, 64, 4, 128, 7, 4}, {128, 32, 32, 64, 8, 128, 7, 4},
    {128, 32, 32, 128, 2, 256, 4, 1}, {128, 64, 16, 128, 4, 256, 4, 2}, {64, 16, 16, 32, 2, 128, 5, 8},
    {128, 32, 32, 32, 2, 128, 4, 1}, {128, 16, 8, 16, 8, 128, 3, 8}, {128, 256, 128, 256, 8, 256, 3, 8},
    {64, 256, 8, 256, 8, 256, 3, 8}, {128, 32, 32, 128, 2, 256, 40, 1}};
  for (auto& c : cfgs)
  for (int tc = 0; tc < 2; ++tc) {
    if (tc && (c[0] != 128 || c[1] < 32)) continue;  // the tensor-core forms' shapes
    PagedArgs a{};
    a.d = c[0]; a.G = c[1]; a.Gv = c[2]; a.R = c[3]; a.bits = c[4]; a.P = c[5]; a.max_pages = c[6];
    a.h_kv = 3; a.n_pages = a.max_pages * 2 + 1; int gq = c[7]; int d = a.d;
    if (tc) {  // the tile choice of the paged tensor-core plan
      for (int t = 256; t >= 32 && !a.tile_pp; t >>= 1)
        if (a.P % t == 0 && tc_fits(t, a.bits, a.bits, d, a.G, a.Gv)) a.tile_pp = t;
      for (int t = 32; t >= 16 && !a.tile_mix; t >>= 1)
        if (t <= a.tile_pp && tc_fits(t, 16, 16, d, a.G, a.Gv) && tc_fits(t, a.bits, 16, d, a.G, a.Gv) &&
            tc_fits(t, 16, a.bits, d, a.G, a.Gv))
          a.tile_mix = t;
    } else {
      for (int t = 128; t >= 16 && !a.tile_pp; t >>= 1) if (fits(t, a.bits, a.bits, d, a.G, a.Gv, gq)) a.tile_pp = t;
      for (int t = a.tile_pp; t >= 16 && !a.tile_mix; t >>= 1)
        if (fits(t, 16, 16, d, a.G, a.Gv, gq) && fits(t, a.bits, 16, d, a.G, a.Gv, gq) && fits(t, 16, a.bits, d, a.G, a.Gv, gq)) a.tile_mix = t;
    }
    const uint32_t cap_bytes = tc ? (uint32_t)kTcStageBytes : (uint32_t)kStageBytes;
    // fake buffers: base addresses far apart, 256-aligned
    const size_t rows = (size_t)a.n_pages * a.h_kv * a.P; const int rb = d * a.bits / 8;
    uintptr_t base = 1ull << 40; auto nb = [&](size_t bytes) { uintptr_t r = base; base += (bytes + 4096) & ~(uintptr_t)255; return r; };
    a.kc = (const uint8_t*)nb(rows * rb); a.vc = (const uint8_t*)nb(rows * rb);
    a.ks = (const __half*)nb(rows / a.G * d * 2); a.kz = (const __half*)nb(rows / a.G * d * 2);
    a.vs = (const __half*)nb(rows * (d / a.Gv) * 2); a.vz = (const __half*)nb(rows * (d / a.Gv) * 2);
    const int B = 2; const size_t ringb = (size_t)B * a.h_kv * a.R * d * 2;
    a.kr = (const __half*)nb(ringb); a.vr = (const __half*)nb(ringb);
    const int cap = a.P * a.max_pages;
    printf("cfg d%d G%d Gv%d R%d b%d P%d %s tile_pp %d tile_mix %d\n", d, a.G, a.Gv, a.R, a.bits, a.P,
           tc ? "tensor-core" : "general", a.tile_pp, a.tile_mix);
    if (!a.tile_pp || !a.tile_mix || a.P % a.tile_pp || a.tile_pp % a.tile_mix) { printf("BAD tiles\n"); bad++; continue; }
    for (int nk = 0; nk <= cap; nk += a.G)
      for (int nkr = 0; nkr <= a.R; ++nkr)
        for (int nvr = 0; nvr <= a.R; nvr += (nvr < 3 || nvr > a.R - 3) ? 1 : 7) {
          const int nv = nk + nkr - nvr;
          if (nv < 0 || nv > cap) continue;
          PagedSeq s{}; s.nk = nk; s.nv = nv; s.nkr = nkr; s.nvr = nvr;
          s.krs = (nk * 7 + 3) % a.R; s.vrs = (nv * 5 + 1) % a.R;
          const int L = nk + nkr, T = paged_tiles(a, s);
          int pos = 0;
          for (int t = 0; t < T; ++t) {
            TileInfo ti = paged_tile(a, s, t);
            ++checked;
            int start = ti.kseg == 0 ? ti.ku0 : ti.ku0 + nk;
            int vstart = ti.vseg == 0 ? ti.vu0 : ti.vu0 + nv;
            bool ok = ti.n >= 1 && ti.n <= (tc ? 256 : 128) && start == pos && vstart == pos && ti.bytes <= cap_bytes;
            if (tc && ti.kseg == 0 &&
                (ti.ng > kTcMaxGroups || (ti.ku0 % 32 != 0 && ti.ku0 / 32 != (ti.ku0 + ti.n - 1) / 32)))
              ok = false;
            if (ti.kseg == 0 && (ti.ku0 / a.P != (ti.ku0 + ti.n - 1) / a.P || ti.ku0 + ti.n > nk)) ok = false;
            if (ti.vseg == 0 && (ti.vu0 / a.P != (ti.vu0 + ti.n - 1) / a.P || ti.vu0 + ti.n > nv)) ok = false;
            if (ti.kseg != 0 && ti.ku0 + ti.n > nkr) ok = false;
            if (ti.vseg != 0 && ti.vu0 + ti.n > nvr) ok = false;
            for (int b = 0; b < B; ++b) for (int h = 0; h < a.h_kv; ++h) {
              uint32_t sum = 0;
              auto page = [&](int row) { return (row / a.P * 5 + b) % a.n_pages; };
              for_each_paged_copy(a, b, h, s, ti, page, [&](const void* src, uint32_t off, uint32_t bytes, int slot) {
                if (slot < 0 || slot > 5) ok = false;
                sum += bytes;
                if (bytes % 16 || off % 16 || ((uintptr_t)src & 15)) ok = false;
                if (off + bytes > ti.bytes) ok = false;
                uintptr_t p = (uintptr_t)src;
                auto in = [&](const void* b0, size_t n) { return p >= (uintptr_t)b0 && p + bytes <= (uintptr_t)b0 + n; };
                if (!(in(a.kc, rows * rb) || in(a.vc, rows * rb) || in(a.ks, rows / a.G * d * 2) || in(a.kz, rows / a.G * d * 2) ||
                      in(a.vs, rows * (d / a.Gv) * 2) || in(a.vz, rows * (d / a.Gv) * 2) || in(a.kr, ringb) || in(a.vr, ringb))) ok = false;
              });
              if (sum != ti.bytes) ok = false;
            }
            if (!ok) { if (bad < 10) printf("BAD nk %d nv %d nkr %d nvr %d t %d n %d\n", nk, nv, nkr, nvr, t, ti.n); ++bad; }
            pos += ti.n;
          }
          if (pos != L) { if (bad < 10) printf("BAD cover nk %d nkr %d nvr %d: %d != %d\n", nk, nkr, nvr, pos, L); ++bad; }
        }
  }
  printf("checked %lld tiles, bad %lld\n", checked, bad);
  return bad != 0;
}
