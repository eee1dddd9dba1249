// CPU replay of the training step's shared blocked copies for one geometry.  When the step
// shares copies, the weight gradient reads x through the forward pass's copy and gradOutput
// through the backward-data pass's copy at a row offset.  This program checks those reads
// against the definition of what the weight gradient needs, element by element:
//   x plane (n, g, chunk j), row q of Rx*Wp:      x[n][g*Cgi + 64j + e][q/Wp - pt][q%Wp - pl]
//   gradOutput plane (n, g, j), row q of Ho*Wp:   dy[n][g*Cgo + 64j + e][q/Wp][q%Wp] (q%Wp < Wo)
// (zero outside the image and past the group's channels), plus the workspace layout: the
// regions are disjoint, 256-byte aligned and inside the reported size, and the gradOutput
// tensor map's base stays 128-byte aligned.  Host code only: the library source is included
// and the few device-facing helpers it calls are stubbed.
// Usage: step_plan_replay <14 or 16 geometry ints> <expect_shared 0|1>
#include "../../bwd_gconv_fwd_gb300/csrc/tc_conv.cu"
#include <cstdio>
#include <cstdlib>
namespace gconv {
long long wait_limit() { return 1000000000LL; }
int num_sms() { return 152; }
unsigned int *device_error_word() { return nullptr; }
int forced_path() { return 0; }
int wgrad_tma_enabled() { return 1; }
void *debug_trace(size_t *b) { *b = 0; return nullptr; }
bool encode_rows_tmap(CUtensorMap *, const void *, uint64_t, uint64_t, uint32_t, uint64_t) { return false; }
}
using namespace gconv;
static long errors = 0;
#define CHECK(cond, ...) do { if (!(cond)) { if (errors++ < 10) { printf("FAIL: " __VA_ARGS__); printf("\n"); } } } while (0)

// What element (plane row q, channel slot e of chunk j) of a blocked copy holds, from the
// copy's parameters alone: the source (channel, row, column), or channel -1 for zero.
struct Src { int ch, r, c; };
static Src copy_element(const BlockifyParams &b, int j, int e, int64_t q)
{
    const int r = (int)(q / b.C), c = (int)(q % b.C);
    const int row = r + b.r_off, col = c + b.c_off;
    const int ch = 64 * j + e;
    if (row < 0 || row >= b.IH || col < 0 || col >= b.IW || ch >= b.Cg) return {-1, 0, 0};
    return {ch, row, col};
}

int main(int argc, char **argv)
{
    int v[16];
    int expect;
    if (argc == 16) {
        int a[14];
        for (int i = 0; i < 14; ++i) a[i] = atoi(argv[1 + i]);
        const int e[16] = {a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], a[7], a[8], a[9], a[10], a[11], a[12], a[12], a[13]};
        for (int i = 0; i < 16; ++i) v[i] = e[i];
        expect = atoi(argv[15]);
    } else if (argc == 18) {
        for (int i = 0; i < 16; ++i) v[i] = atoi(argv[1 + i]);
        expect = atoi(argv[17]);
    } else {
        printf("usage: step_plan_replay <14 or 16 geometry ints> <expect_shared>\n");
        return 2;
    }
    const int span_h = v[2] + v[9] + v[10] - v[13] * (v[5] - 1) - 1, span_w = v[3] + v[11] + v[12] - v[14] * (v[6] - 1) - 1;
    Geom g{v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15],
           span_h / v[7] + 1, span_w / v[8] + 1, v[1] / v[15], v[4] / v[15]};
    TcStep S;
    const bool shared = tc_step_build(g, &S);
    printf("shared=%d y_off=%lld ws=%zu\n", (int)shared, (long long)S.y_off, S.ws_bytes);
    CHECK(shared == (expect != 0), "shared route %d, expected %d", (int)shared, expect);
    if (shared) {
        const WgradParams &w = S.W.wp;
        const BlockifyParams &fx = S.F.bu, &by = S.B.bu;
        // x: the forward copy's planes are the weight gradient's, row for row
        CHECK((int64_t)fx.R * fx.C == (int64_t)w.Rx * w.Wp, "x plane %d x %d against %d x %d", fx.R, fx.C, w.Rx, w.Wp);
        CHECK(fx.nchunk == w.ncx && fx.Cg == g.Cgi && fx.N == g.N && fx.G == g.G, "x planes");
        for (int j = 0; j < w.ncx; ++j)
            for (int e = 0; e < 64; e += 7)
                for (int64_t q = 0; q < (int64_t)w.Rx * w.Wp; ++q) {
                    const Src a = copy_element(fx, j, e, q);
                    const int r = (int)(q / w.Wp) - g.pt, c = (int)(q % w.Wp) - g.pl, ch = 64 * j + e;
                    const bool in = r >= 0 && r < g.H && c >= 0 && c < g.W && ch < g.Cgi;
                    CHECK(in ? (a.ch == ch && a.r == r && a.c == c) : a.ch < 0,
                          "x chunk %d slot %d row %lld: copy (%d,%d,%d)", j, e, (long long)q, a.ch, a.r, a.c);
                }
        // the ones slot sits past the valid channels of the last chunk, where the forward
        // pass's packed weights are zero
        CHECK(S.W.ones < 0 || (S.W.ones == g.Cgi % 64 && 64 * (w.ncx - 1) + S.W.ones >= g.Cgi), "ones slot");
        // gradOutput: the weight gradient's plane row q is the backward copy's row y_off + q
        CHECK(by.nchunk == w.ncy && by.Cg == g.Cgo, "gradOutput planes");
        const int64_t bplane = (int64_t)by.R * by.C;
        CHECK(S.y_off >= 0 && S.y_off + (int64_t)w.Ho * w.Wp <= bplane, "gradOutput window past the plane");
        for (int j = 0; j < w.ncy; ++j)
            for (int e = 0; e < 64; e += 5)
                for (int64_t q = 0; q < (int64_t)w.Ho * w.Wp; ++q) {
                    const Src a = copy_element(by, j, e, S.y_off + q);
                    const int r = (int)(q / w.Wp), c = (int)(q % w.Wp), ch = 64 * j + e;
                    const bool in = c < g.Wo && ch < g.Cgo;
                    CHECK(in ? (a.ch == ch && a.r == r && a.c == c) : a.ch < 0,
                          "dy chunk %d slot %d row %lld: copy (%d,%d,%d)", j, e, (long long)q, a.ch, a.r, a.c);
                }
        CHECK((S.y_off * 64 * 2) % 128 == 0, "gradOutput map base alignment");
        // workspace regions: [x copy, forward weights], [gradOutput copy, backward weights],
        // split-K slices, bias slices, in order, disjoint and aligned
        const size_t ends[4] = {S.off_fx + S.F.ub_bytes + S.F.wpk_bytes, S.off_bx + S.B.ub_bytes + S.B.wpk_bytes,
                                S.off_part + S.W.part_bytes, S.off_bias + S.W.bias_bytes};
        const size_t starts[4] = {S.off_fx, S.off_bx, S.off_part, S.off_bias};
        for (int i = 0; i < 4; ++i) {
            CHECK(starts[i] % 256 == 0, "region %d alignment", i);
            CHECK(ends[i] <= S.ws_bytes, "region %d past the workspace", i);
            if (i) CHECK(starts[i] >= ends[i - 1], "regions %d and %d overlap", i - 1, i);
        }
        CHECK(S.F.ub_bytes >= (size_t)g.N * g.G * w.ncx * w.Rx * w.Wp * 128, "x copy size");
        CHECK(S.B.ub_bytes >= (size_t)g.N * g.G * w.ncy * bplane * 128, "gradOutput copy size");
    }
    printf("errors: %ld\n", errors);
    return errors ? 1 : 0;
}
