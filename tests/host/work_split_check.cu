// Host-side brute force over the tensor-core kernels' work split (la_tc_common.cuh), run on the CPU:
// slices tile the chunk list, cta_of inverts them, pieces stay within one head and cover each slice in
// order (RevPieceIter gives them back last first), and the per-piece state slots never collide and fit the workspace's BH + kMaxCtas slots; the
// grid that choose_ctas picks stays within bounds, and where it departs from the default every slice is
// one piece of one head.  Prints "ok <cases>" and exits 0, or prints the first failing case and exits 1.
#include <stdio.h>
#include <stdlib.h>

#include <vector>

#include "la_tc_common.cuh"

using namespace la::tc;

static unsigned long long rng_state = 0x9E3779B97F4A7C15ull;
static unsigned long long next_rand() {  // splitmix64
    unsigned long long z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static int check(long long BH, int nchunk, int G) {
    Slices s;
    s.T = BH * nchunk;
    s.G = G;
    s.nchunk = nchunk;
    if (slice_lo(s, 0) != 0 || slice_lo(s, G) != s.T) return 1;
    for (int b = 0; b < G; ++b)
        if (slice_lo(s, b + 1) <= slice_lo(s, b)) return 2;  // every slice non-empty (G <= T)
    for (int b = 0; b < G; ++b)
        for (long long x = slice_lo(s, b); x < slice_lo(s, b + 1); ++x)
            if (cta_of(s, x) != b) return 3;
    std::vector<char> slot_used((size_t)(BH + kMaxCtas), 0);
    long long covered = 0;
    for (int b = 0; b < G; ++b) {
        long long expect = slice_lo(s, b);
        for (PieceIter pi(s, b); pi.valid(); pi.next()) {
            const Piece p = pi.get();
            if (p.h < 0 || p.h >= BH || p.a < 0 || p.e > nchunk || p.a >= p.e) return 4;
            if (p.h * nchunk + p.a != expect) return 5;  // pieces follow one another without gaps
            expect = p.h * nchunk + p.e;
            covered += p.e - p.a;
            const long long slot = slot_of(p.h, b);
            if (slot < 0 || slot >= BH + kMaxCtas) return 6;
            if (slot_used[(size_t)slot]) return 7;  // two pieces share a slot
            slot_used[(size_t)slot] = 1;
        }
        if (expect != slice_lo(s, b + 1)) return 8;
        // RevPieceIter yields the same pieces, last first
        std::vector<Piece> fwd, rev;
        for (PieceIter pi(s, b); pi.valid(); pi.next()) fwd.push_back(pi.get());
        for (RevPieceIter pi(s, b); pi.valid(); pi.next()) rev.push_back(pi.get());
        if (fwd.size() != rev.size()) return 12;
        for (size_t k = 0; k < fwd.size(); ++k) {
            const Piece &f = fwd[fwd.size() - 1 - k], &r = rev[k];
            if (f.h != r.h || f.a != r.a || f.e != r.e) return 13;
        }
    }
    if (covered != s.T) return 9;
    // the CTAs that cover a head are contiguous, from cta_of(first chunk) to cta_of(last chunk)
    for (long long h = 0; h < BH; ++h) {
        const int b0 = cta_of(s, h * nchunk), b1 = cta_of(s, h * nchunk + nchunk - 1);
        long long n = 0;
        for (int b = b0; b <= b1; ++b) {
            bool has = false;
            for (PieceIter pi(s, b); pi.valid(); pi.next()) has |= pi.get().h == h;
            if (!has) return 10;
            n += 1;
        }
        if (n != b1 - b0 + 1) return 11;
    }
    return 0;
}

int main() {
    // slot_f4 is a permutation of the 4096 float4 of a 128 x 128 slot matrix
    std::vector<char> seen(4096, 0);
    for (int d = 0; d < 128; ++d)
        for (int hf = 0; hf < 2; ++hf)
            for (int q = 0; q < 16; ++q) {
                const long long f = slot_f4(d, hf, q);
                if (f < 0 || f >= 4096 || seen[(size_t)f]) {
                    printf("slot_f4 not a permutation at d=%d hf=%d q=%d\n", d, hf, q);
                    return 1;
                }
                seen[(size_t)f] = 1;
            }
    long long cases = 0;
    // exhaustive over small shapes, then random larger ones (G <= min(T, kMaxCtas), as the launcher sets it)
    for (long long BH = 1; BH <= 12; ++BH)
        for (int nchunk = 1; nchunk <= 12; ++nchunk) {
            const long long T = BH * nchunk;
            for (int G = 1; G <= (T < kMaxCtas ? T : kMaxCtas); ++G, ++cases)
                if (int rc = check(BH, nchunk, G)) {
                    printf("fail %d: BH=%lld nchunk=%d G=%d\n", rc, BH, nchunk, G);
                    return 1;
                }
        }
    for (int t = 0; t < 3000; ++t, ++cases) {
        const long long BH = 1 + (long long)(next_rand() % 512);
        const int nchunk = 1 + (int)(next_rand() % 600);
        const long long T = BH * nchunk;
        const long long gmax = T < kMaxCtas ? T : kMaxCtas;
        const int G = 1 + (int)(next_rand() % (unsigned long long)gmax);
        if (int rc = check(BH, nchunk, G)) {
            printf("fail %d: BH=%lld nchunk=%d G=%d\n", rc, BH, nchunk, G);
            return 1;
        }
    }
    // choose_ctas: within [1, min(T, nsm, kMaxCtas)]; narrow heads get the default; where it departs from
    // the default, every slice is one piece (nchunk / k chunks of one head) and the split itself is valid
    for (long long BH = 1; BH <= 300; BH += (BH < 40 ? 1 : 7))
        for (int nchunk = 1; nchunk <= 600; nchunk += (nchunk < 40 ? 1 : 13))
            for (int nsm : {152, 148, 132, 8})
                for (int causal = 0; causal < 2; ++causal)
                    for (int full = 0; full < 2; ++full, ++cases) {
                        const long long T = BH * nchunk;
                        long long def = T < nsm ? T : nsm;
                        if (def > kMaxCtas) def = kMaxCtas;
                        const long long G = choose_ctas(BH, nchunk, nsm, causal != 0, full != 0);
                        bool bad = G < 1 || G > def || (!full && G != def);
                        if (!bad && G != def) {
                            Slices s;
                            s.T = T;
                            s.G = (int)G;
                            s.nchunk = nchunk;
                            bad = check(BH, nchunk, (int)G) != 0 || (T % G) != 0 || (nchunk % (T / G)) != 0;
                            for (int b = 0; b < G && !bad; ++b) {
                                int pieces = 0;
                                for (PieceIter pi(s, b); pi.valid(); pi.next()) ++pieces;
                                bad = pieces != 1;
                            }
                            // no more chunks per CTA than the default (causal), at most two more (non-causal)
                            bad = bad || (T / G) - (T + def - 1) / def > (causal ? 0 : 2);
                        }
                        if (bad) {
                            printf("choose_ctas fails: BH=%lld nchunk=%d nsm=%d causal=%d full=%d G=%lld\n", BH, nchunk,
                                   nsm, causal, full, G);
                            return 1;
                        }
                    }
    printf("ok %lld\n", cases);
    return 0;
}
