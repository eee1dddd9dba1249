// CPU replay of the correlation kernel's launch plan and index arithmetic for one geometry
// (forward and backward-data): every weight tap used once, paired-tap offsets, staged rows
// within the blocked copy, weight blocks within the packed buffer, TMEM columns of the paired
// epilogue within one accumulator, every store inside the output, every output position
// covered by exactly one tile.  Host code only: the library source is included and the few
// device-facing helpers it calls are stubbed.  Usage: corr2_plan_replay <14 geometry ints>;
// exits non-zero and prints FAIL lines on any violation.
#include "../../bwd_gconv_fwd_gb300/csrc/tc_conv.cu"
#include <cstdio>
#include <cstdlib>
namespace gconv {
long long wait_limit() { return 1000000000LL; }
int num_sms() { return 152; }
unsigned int *device_error_word() { return nullptr; }
int forced_path() { return 0; }
void *debug_trace(size_t *b) { *b = 0; return nullptr; }
bool encode_rows_tmap(CUtensorMap *, const void *, uint64_t, uint64_t, uint32_t) { return false; }
}
using namespace gconv;
static long errors = 0;
#define CHECK(cond, ...) do { if (!(cond)) { if (errors++ < 10) { printf("FAIL: " __VA_ARGS__); printf("\n"); } } } while (0)
int main(int argc, char **argv)
{
    // 14 geometry integers (one stride, one dilation) or 16 (per axis)
    int v[16];
    if (argc == 15) {
        int a[14];
        for (int i = 0; i < 14; ++i) a[i] = atoi(argv[1 + i]);
        const int e[16] = {a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], a[7], a[8], a[9], a[10], a[11], a[12], a[12], a[13]};
        for (int i = 0; i < 16; ++i) v[i] = e[i];
    } else {
        for (int i = 0; i < 16; ++i) v[i] = atoi(argv[1 + i]);
    }
    const int span_h = v[2] + v[9] + v[10] - v[13] * (v[5] - 1) - 1, span_w = v[3] + v[11] + v[12] - v[14] * (v[6] - 1) - 1;
    Geom g{v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15],
           span_h / v[7] + 1, span_w / v[8] + 1, v[1] / v[15], v[4] / v[15]};
    for (int bd = 0; bd < 2; ++bd) {
        Corr2Launch C;
        if (!build_corr2(g, bd == 1, &C)) { printf("corr2 %d not served\n", bd); continue; }
        const Corr2Params &c = C.cp;
        const Pack2Params &k = C.pk;
        printf("corr2 bwd_data=%d: Cv=%d pair_delta=%d nmma=%d tile_pos=%d blocks=%d stage_rows=%d tiles=%d smem=%zu\n", bd, c.Cv,
               c.pair_delta, c.nmma, c.tile_pos, c.ntaps, c.stage_rows, c.n_tiles, C.smem);
        // every weight tap used exactly once
        std::vector<int> seen(g.kH * g.kW, 0);
        for (int b = 0; b < c.ntaps; ++b) {
            seen[k.tk1[b]]++;
            if (k.tk2[b] >= 0) seen[k.tk2[b]]++;
            CHECK(c.tap_off[b] + c.nmma <= c.stage_rows, "B rows");
        }
        for (size_t t = 0; t < seen.size(); ++t) CHECK(seen[t] == 1, "tap %zu used %d times", t, seen[t]);
        // pair semantics: second tap offset = first + pair_delta (recomputed from the tap indices)
        for (int b = 0; b < c.ntaps; ++b)
            if (k.tk2[b] >= 0) {
                auto off = [&](int t) { const int kh = t / g.kW, kw = t % g.kW;
                    const int a = bd ? (g.kH - 1 - kh) * g.d_h : kh * g.d_h, bb = bd ? (g.kW - 1 - kw) * g.d_w : kw * g.d_w; return a * c.Wp + bb; };
                CHECK(off(k.tk1[b]) == c.tap_off[b] && off(k.tk2[b]) == c.tap_off[b] + c.pair_delta, "pair offsets");
                CHECK(c.Cv <= 64 && c.n_vtile == 1, "pair needs one 64-row half");
            }
        // TMEM columns read by the epilogue stay in the 256-column buffer
        if (c.pair_delta) {
            int maxcol = 0;
            for (int pc = 0; pc < c.tile_pos; pc += 16) maxcol = std::max(maxcol, pc + c.pair_delta + 15);
            CHECK(maxcol <= 255, "upper TMEM column %d", maxcol);
        }
        const int plane = c.R * c.Wp;
        const size_t out_elems = (size_t)c.N * c.G * c.Cv * c.Qh * c.Qw;
        const int64_t out_hw = (int64_t)c.Qh * c.Qw;
        for (int t = 0; t < c.n_tiles; ++t) {
            int tt = t;
            const int ptile = tt % c.n_ptile; tt /= c.n_ptile;
            const int n = tt % c.N; tt /= c.N;
            const int vt = tt % c.n_vtile;
            const int gg = tt / c.n_vtile;
            const int p0 = ptile * c.tile_pos;
            for (int kc = 0; kc < c.nchu; ++kc)
                for (int m = 0; m < c.stage_rows; ++m)
                    if (p0 + m < plane) {
                        const int64_t e = ((((int64_t)n * c.G + gg) * c.nchu + kc) * plane + p0 + m) * 64;
                        CHECK((size_t)(e + 64) * 2 <= C.ub_bytes, "stage src");
                    }
            CHECK((((size_t)gg * c.n_vtile + vt) + 1) * c.nchu * c.ntaps * kWblkBytes <= C.wpk_bytes, "weights");
            // stores: each tile writes positions [p0, p0 + tile_pos) that are real outputs
            const int cols = c.tile_pos;
            for (int j = 0; j < cols; ++j) {
                const int pos = p0 + j, qh = pos / c.Wp, qw = pos % c.Wp;
                if (!(qh < c.Qh && qw < c.Qw)) continue;
                for (int vv = 0; vv < std::min(c.Cv, 128); ++vv) {
                    const int64_t e = ((int64_t)n * c.G * c.Cv + (int64_t)gg * c.Cv + vt * 128 + vv) * out_hw + (int64_t)qh * c.Qw + qw;
                    CHECK(e >= 0 && (size_t)e < out_elems, "store");
                }
            }
        }
        // coverage: every real output position belongs to exactly one tile
        std::vector<int> cov(plane, 0);
        for (int pt = 0; pt < c.n_ptile; ++pt)
            for (int j = 0; j < c.tile_pos; ++j) if (pt * c.tile_pos + j < plane) cov[pt * c.tile_pos + j]++;
        for (int pos = 0; pos < c.Qh * c.Wp; ++pos) if (pos % c.Wp < c.Qw) CHECK(cov[pos] == 1, "coverage %d: %d", pos, cov[pos]);
    }
    printf("errors: %ld\n", errors);
    return errors ? 1 : 0;
}
