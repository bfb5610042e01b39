// schedule_harness.cu -- host program that prints the attention kernels'
// tile schedule (round_span for the forward, query_span for the backward,
// from the kernels' own header) for one problem, so a CPU test can compare
// it tile by tile with the oracle's causal mask on the positions of each
// placement.  Built and run by tests/test_schedule_host.py; no GPU needed.
//
// usage: schedule_harness LAYOUT S N T
// prints "R d e a nfull has_diag diag_off" for every query tile a of every
// (device d, key stripe e), then "Q d e b a_lo has_diag diag_off" for every
// key tile b.
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"

int main(int argc, char **argv) {
    if (argc != 5) {
        fprintf(stderr, "usage: %s LAYOUT S N T\n", argv[0]);
        return 2;
    }
    const int layout = atoi(argv[1]);
    const long S = atol(argv[2]);
    const int N = atoi(argv[3]);
    const int T = atoi(argv[4]);
    if (N < 1 || T < 1 || S % N != 0) return 2;
    const long L = S / N;
    const int n = (int)((L + T - 1) / T);  // tiles per stripe (queries and keys alike)
    for (int d = 0; d < N; ++d)
        for (int e = 0; e < N; ++e)
            for (int a = 0; a < n; ++a) {
                const long rows = L - (long)a * T;
                const striped::RoundSpan s = striped::round_span(layout, d, e, a, n, rows >= T ? T : (int)rows);
                printf("R %d %d %d %d %d %d\n", d, e, a, s.nfull, s.has_diag, s.diag_off);
            }
    for (int d = 0; d < N; ++d)
        for (int e = 0; e < N; ++e)
            for (int b = 0; b < n; ++b) {
                const long rows = L - (long)b * T;
                const striped::QuerySpan s = striped::query_span(layout, d, e, b, n, rows >= T ? T : (int)rows);
                printf("Q %d %d %d %d %d %d\n", d, e, b, s.a_lo, s.has_diag, s.diag_off);
            }
    return 0;
}
