#include <algorithm>
#include <cstdio>
#include <utility>
#include <vector>
// Host enumeration of the one-query-head decode kernel's chunk geometry
// (kvq_internal.h: warp_chunk, warp_piece_start, warp_chunk_copies) over
// many cache states, ring starts and pair counts: the chunks cover [0, L) in
// token order (32-token chunks where K and V are packed, 8-token blocks
// elsewhere), the pieces of a pair cut into k or k - 1 cover its chunks in
// order and none is empty, and every copy of every chunk of the first and
// the last pair is 16-byte aligned, inside its buffer, inside the slot and
// disjoint from the chunk's other copies.  Built and run on the CPU by
// tests/test_plan_cpu.py; exits nonzero on a bad chunk.
#include "../quantized_kv_cache_kivi_gb300/csrc/kvq_internal.h"
using namespace kvq;

int main() {
  long long checked = 0, bad = 0;
  const int Gs[] = {32, 64, 128}, Gvs[] = {32, 64, 128}, Rs[] = {64, 128, 256}, caps[] = {256, 1024, 4224};
  const int Ps[] = {1, 7, 2048};
  for (int G : Gs)
    for (int Gv : Gvs)
      for (int R : Rs) {
        if (R % G) continue;
        for (int cap : caps) {
          if (cap % G || cap % 32) continue;
          for (int nk = 0; nk <= cap; nk += (nk < 256 ? G : 7 * G)) {
            for (int nkr : {0, 1, 7, R / 2, R - 1, R}) {
              const int L = nk + nkr;
              if (L == 0) continue;
              for (int nvr : {0, 1, 9, R / 2 + 1, R}) {
                if (nvr > L) continue;
                const int nv = L - nvr;
                if (nv > cap || nk % 8) continue;
                for (int rs : {0, 3, R - 1}) {
                  WarpArgs a{};
                  a.cap = cap;
                  a.R = R;
                  a.krs = rs;
                  a.vrs = (rs * 5 + 1) % R;
                  a.log2G = 0;
                  while ((1 << a.log2G) < G) ++a.log2G;
                  a.ngv = 128 / Gv;
                  a.nk = nk;
                  a.nv = nv;
                  a.L = L;
                  a.npp = std::min(nk, nv);
                  a.npx = std::max(nk, nv);
                  a.n_pp = (a.npp + 31) / 32;
                  a.n_x1 = a.npx > a.npp ? (a.npx - 1) / 8 - a.npp / 8 + 1 : 0;
                  a.n_x2 = a.L > a.npx ? (a.L - 1) / 8 - a.npx / 8 + 1 : 0;
                  a.C = a.n_pp + a.n_x1 + a.n_x2;
                  a.Cp = (long long)kWarpWpp * a.n_pp + (long long)kWarpWx * (a.n_x1 + a.n_x2);
                  // chunks: contiguous cover of [0, L)
                  int next = 0;
                  for (int c = 0; c < a.C; ++c) {
                    const WarpChunk ch = warp_chunk(a, c);
                    ++checked;
                    const int lim = ch.pp ? 32 : 8;
                    if (ch.t0 != next || ch.n < 1 || ch.o0 < 0 || ch.o0 + ch.n > lim || (ch.pp && ch.o0 != 0) ||
                        ch.kq != (ch.t0 < nk) || ch.vq != (ch.t0 < nv) ||
                        (ch.t0 + ch.n > nk && ch.t0 < nk) || (ch.t0 + ch.n > nv && ch.t0 < nv)) {
                      if (bad++ < 10)
                        printf("bad chunk: G %d R %d nk %d nkr %d nv %d c %d t0 %d n %d o0 %d\n", G, R, nk, nkr, nv, c,
                               ch.t0, ch.n, ch.o0);
                    }
                    next = ch.t0 + ch.n;
                  }
                  if (next != L && bad++ < 10) printf("chunks end at %d, not %d\n", next, L);
                  // pieces: k and k - 1 per pair, none empty
                  const long long kmax = std::min<long long>(16, a.Cp / std::max(kWarpWpp, kWarpWx));
                  for (long long k = 1; k <= kmax; ++k)
                    for (long long kp = k - 1; kp <= k; ++kp) {
                      if (kp < 1) continue;
                      a.k = (int)k;
                      if (warp_piece_start(a, (int)kp, 0) != 0 || warp_piece_start(a, (int)kp, (int)kp) != a.C) ++bad;
                      for (int j = 0; j < kp; ++j)
                        if (warp_piece_start(a, (int)kp, j + 1) <= warp_piece_start(a, (int)kp, j)) {
                          if (bad++ < 10) printf("empty piece: Cp %lld kp %lld j %d\n", a.Cp, kp, j);
                        }
                    }
                  // copies of the first and the last pair
                  for (int P : Ps) {
                    const size_t rows = (size_t)P * cap;
                    const uintptr_t b0 = (uintptr_t)1 << 40;
                    uintptr_t base[8];
                    const size_t ext[8] = {rows * 32,
                                           (size_t)P * (cap / G) * 256,
                                           (size_t)P * (cap / G) * 256,
                                           rows * 32,
                                           rows * a.ngv * 2,
                                           rows * a.ngv * 2,
                                           (size_t)P * R * 256,
                                           (size_t)P * R * 256};
                    uintptr_t at = b0;
                    for (int i = 0; i < 8; ++i) {
                      base[i] = at;
                      at += (ext[i] + 4095) / 4096 * 4096 + 4096;
                    }
                    a.kc = reinterpret_cast<const uint8_t*>(base[0]);
                    a.ks = reinterpret_cast<const __half*>(base[1]);
                    a.kz = reinterpret_cast<const __half*>(base[2]);
                    a.vc = reinterpret_cast<const uint8_t*>(base[3]);
                    a.vs = reinterpret_cast<const __half*>(base[4]);
                    a.vz = reinterpret_cast<const __half*>(base[5]);
                    a.kr = reinterpret_cast<const __half*>(base[6]);
                    a.vr = reinterpret_cast<const __half*>(base[7]);
                    for (long long pair : {0LL, (long long)P - 1}) {
                      for (int c = 0; c < a.C; ++c) {
                        const WarpChunk ch = warp_chunk(a, c);
                        std::vector<std::pair<uint32_t, uint32_t>> iv;
                        bool ok = true;
                        warp_chunk_copies(a, pair, ch, [&](const void* src, uint32_t dst, uint32_t n, int buf) {
                          const uintptr_t p = reinterpret_cast<uintptr_t>(src);
                          if (n == 0 || n % 16 || p % 16 || dst % 16 || dst + n > (uint32_t)kWarpSlot ||
                              p < base[buf] || p + n > base[buf] + ext[buf])
                            ok = false;
                          iv.push_back({dst, dst + n});
                        });
                        std::sort(iv.begin(), iv.end());
                        for (size_t i = 1; i < iv.size(); ++i)
                          if (iv[i].first < iv[i - 1].second) ok = false;
                        if (!ok && bad++ < 10)
                          printf("bad copy: G %d Gv %d R %d cap %d nk %d nkr %d nv %d P %d pair %lld c %d\n", G, Gv, R,
                                 cap, nk, nkr, nv, P, pair, c);
                      }
                    }
                  }
                }
              }
            }
          }
        }
      }
  printf("checked %lld chunks, bad %lld\n", checked, bad);
  return bad ? 1 : 0;
}
