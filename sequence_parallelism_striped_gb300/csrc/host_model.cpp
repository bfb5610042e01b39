// host_model.cpp -- exact per-round tile table and modelled ring critical
// path (host only; declared in include/striped.h).
//
// Ring rounds: in round r virtual device d holds the key/value stripe of
// device e = (d - r) mod N (research.elamur.ai summary page, §Summary).  A
// query tile (rows [i0, i1) of stripe d) and key tile (rows [j0, j1) of
// stripe e) is counted when at least one of its pairs is kept, "full" when
// all are.  Pair (i, j) is kept iff the key position <= the query position:
//   striped    (row d*L+i holds i*N+d):  j <= i + c,  c = [e <= d] - 1
//   contiguous (row d*L+i holds d*L+i):  e < d: all;  e == d: j <= i;
//                                        e > d: none.
//   zig-zag (row d*L+i holds d*C+i for i < C, (2N-1-d)*C+i-C otherwise,
//            C = S/(2N)): compare the positions directly.
// For "j <= i + c" a tile has a kept pair iff j0 <= (i1 - 1) + c and all
// pairs kept iff (j1 - 1) <= i0 + c; in general, since positions grow with
// the row inside a device, a tile has a kept pair iff pos(j0) <= pos(i1-1)
// and all pairs kept iff pos(j1-1) <= pos(i0).  Each tile is classified in
// O(1).
// Critical path: each round lasts as long as its busiest device (§Summary:
// rounds run at the pace of the slowest device), summed over rounds.
#include <stdint.h>
#include <stdlib.h>

#include "striped.h"

namespace {

// Zig-zag position of row i of device d (C = L / 2 positions per chunk).
inline int64_t zigzag_pos(int64_t d, int64_t i, int64_t C, int N) {
    return i < C ? d * C + i : (2 * (int64_t)N - 1 - d) * C + (i - C);
}

// class of one tile: 0 = skipped, 1 = full, 2 = partial
inline int classify(int layout, int N, int64_t L, int d, int e, int64_t i0, int64_t i1, int64_t j0,
                    int64_t j1) {
    if (layout == STRIPED_LAYOUT_ZIGZAG) {
        const int64_t C = L / 2;
        if (zigzag_pos(e, j0, C, N) > zigzag_pos(d, i1 - 1, C, N)) return 0;
        if (zigzag_pos(e, j1 - 1, C, N) <= zigzag_pos(d, i0, C, N)) return 1;
        return 2;
    }
    int64_t c;
    if (layout == STRIPED_LAYOUT_STRIPED) {
        c = (e <= d) ? 0 : -1;
    } else {
        if (e < d) return 1;
        if (e > d) return 0;
        c = 0;
    }
    if (j0 > (i1 - 1) + c) return 0;
    if ((j1 - 1) <= i0 + c) return 1;
    return 2;
}

}  // namespace

extern "C" {

int striped_tile_counts(int64_t S, int N, int Tq, int Tk, int layout, int64_t *full, int64_t *partial) {
    if (S < 1 || N < 1 || Tq < 1 || Tk < 1 || S % N != 0) return STRIPED_ERR_INVALID_ARG;
    if (layout != STRIPED_LAYOUT_STRIPED && layout != STRIPED_LAYOUT_CONTIGUOUS && layout != STRIPED_LAYOUT_ZIGZAG)
        return STRIPED_ERR_INVALID_ARG;
    if (layout == STRIPED_LAYOUT_ZIGZAG && S % (2 * (int64_t)N) != 0) return STRIPED_ERR_INVALID_ARG;
    const int64_t L = S / N;
    for (int r = 0; r < N; ++r) {
        for (int d = 0; d < N; ++d) {
            const int e = ((d - r) % N + N) % N;
            int64_t nf = 0, np = 0;
            for (int64_t i0 = 0; i0 < L; i0 += Tq) {
                const int64_t i1 = (i0 + Tq < L) ? i0 + Tq : L;
                for (int64_t j0 = 0; j0 < L; j0 += Tk) {
                    const int64_t j1 = (j0 + Tk < L) ? j0 + Tk : L;
                    const int k = classify(layout, N, L, d, e, i0, i1, j0, j1);
                    if (k == 0) {
                        // key positions grow with j, so later key tiles are masked too
                        break;
                    }
                    if (k == 1) ++nf;
                    else ++np;
                }
            }
            if (full) full[r * N + d] = nf;
            if (partial) partial[r * N + d] = np;
        }
    }
    return STRIPED_OK;
}

// Packed sequences: each sequence is placed and tiled on its own, so a
// device's work in round r is the sum of the sequences' tables.
int striped_tile_counts_varlen(const int32_t *cu_seqlens, int nseq, int N, int Tq, int Tk, int layout,
                               int64_t *full, int64_t *partial) {
    if (!cu_seqlens || nseq < 1 || N < 1 || N > 4096 || cu_seqlens[0] != 0) return STRIPED_ERR_INVALID_ARG;
    const size_t nn = (size_t)N * N;
    int64_t *f = (int64_t *)malloc(sizeof(int64_t) * nn);
    int64_t *p = (int64_t *)malloc(sizeof(int64_t) * nn);
    if (!f || !p) {
        free(f);
        free(p);
        return STRIPED_ERR_INVALID_ARG;
    }
    for (size_t x = 0; x < nn; ++x) {
        if (full) full[x] = 0;
        if (partial) partial[x] = 0;
    }
    int st = STRIPED_OK;
    for (int i = 0; i < nseq && st == STRIPED_OK; ++i) {
        const int64_t len = (int64_t)cu_seqlens[i + 1] - cu_seqlens[i];
        if (len <= 0) {
            st = STRIPED_ERR_INVALID_ARG;
            break;
        }
        st = striped_tile_counts(len, N, Tq, Tk, layout, f, p);
        for (size_t x = 0; x < nn && st == STRIPED_OK; ++x) {
            if (full) full[x] += f[x];
            if (partial) partial[x] += p[x];
        }
    }
    free(f);
    free(p);
    return st;
}

int64_t striped_critical_path_varlen(const int32_t *cu_seqlens, int nseq, int N, int Tq, int Tk, int layout) {
    if (N < 1 || N > 4096) return STRIPED_ERR_INVALID_ARG;
    const size_t nn = (size_t)N * N;
    int64_t *f = (int64_t *)malloc(sizeof(int64_t) * nn);
    int64_t *p = (int64_t *)malloc(sizeof(int64_t) * nn);
    if (!f || !p) {
        free(f);
        free(p);
        return STRIPED_ERR_INVALID_ARG;
    }
    int64_t total = striped_tile_counts_varlen(cu_seqlens, nseq, N, Tq, Tk, layout, f, p);
    if (total == STRIPED_OK) {
        for (int r = 0; r < N; ++r) {
            int64_t mx = 0;
            for (int d = 0; d < N; ++d) {
                const int64_t c = f[r * N + d] + p[r * N + d];
                if (c > mx) mx = c;
            }
            total += mx;
        }
    }
    free(f);
    free(p);
    return total;
}

int64_t striped_critical_path(int64_t S, int N, int Tq, int Tk, int layout) {
    if (N < 1 || N > 4096) return STRIPED_ERR_INVALID_ARG;
    int64_t *f = (int64_t *)malloc(sizeof(int64_t) * (size_t)N * N);
    int64_t *p = (int64_t *)malloc(sizeof(int64_t) * (size_t)N * N);
    if (!f || !p) {
        free(f);
        free(p);
        return STRIPED_ERR_INVALID_ARG;
    }
    int st = striped_tile_counts(S, N, Tq, Tk, layout, f, p);
    int64_t total = st;
    if (st == STRIPED_OK) {
        total = 0;
        for (int r = 0; r < N; ++r) {
            int64_t mx = 0;
            for (int d = 0; d < N; ++d) {
                const int64_t c = f[r * N + d] + p[r * N + d];
                if (c > mx) mx = c;
            }
            total += mx;
        }
    }
    free(f);
    free(p);
    return total;
}

}  // extern "C"
