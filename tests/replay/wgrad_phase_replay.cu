// CPU replay of the stride-2 weight-gradient launch plan and index arithmetic for one
// geometry: the stride-phase blocked copy's reads and writes, the one launch's job groups
// (rows and TMEM columns; each group reads its own x phase plane), every staged gradOutput
// and input row within its buffer and phase plane, every split-K partial within the
// workspace, every tap covered by exactly one job.  Host
// code only (library source included, device-facing helpers stubbed).  Usage:
// wgrad_phase_replay <14 geometry ints>; exits non-zero and prints FAIL lines on a violation.
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
    WgradPhaseLaunch L;
    if (!build_wgrad_phases(g, &L)) { printf("not served by this path\nerrors: 0\n"); return 0; }
    printf("Ho=%d Wo=%d nphase=%d xplane_elems=%zu ws=%zu\n", g.Ho, g.Wo, L.nphase, L.xplane_elems, L.ws_bytes);
    // phase blocked copy
    {
        const PhaseBlockifyParams &p = L.bx;
        const int plane_out = p.R * p.C;
        const int64_t ngj = (int64_t)p.N * p.G * p.nchunk;
        const int64_t total = ngj * p.nplane * plane_out;
        const size_t in_elems = (size_t)g.N * g.Cin * g.H * g.W;
        for (int64_t q = 0; q < total; ++q) {
            const int64_t blk = q / plane_out;
            const int pos = (int)(q - blk * plane_out);
            const int r = pos / p.C, c = pos - r * p.C;
            const int j = (int)(blk % p.nchunk);
            const int64_t t = blk / p.nchunk;
            const int64_t ng = t % ((int64_t)p.N * p.G);
            const int pl = (int)(t / ((int64_t)p.N * p.G));
            const int row = r * p.s_h + p.roff[pl], col = c * p.s_w + p.coff[pl];
            const bool inside = row >= 0 && row < p.IH && col >= 0 && col < p.IW;
            const int cvalid = inside ? std::min(64, p.Cg - 64 * j) : 0;
            const int64_t plane = (int64_t)p.IH * p.IW;
            const int64_t base = (ng * p.Cg + 64 * j) * plane + (inside ? (int64_t)row * p.IW + col : 0);
            for (int e = 0; e < cvalid; ++e) CHECK((size_t)(base + e * plane) < in_elems, "bx src");
            CHECK((size_t)(q * 8 + 8) * 16 <= L.xt_bytes, "bx dst");
            // phase semantics: plane pl row r holds x row (r + row0)*s + ph
        }
    }
    const size_t xt_elems = L.xt_bytes / 2, yt_elems = L.yt_bytes / 2, part_elems = L.part_bytes / 4;
    std::vector<int> tap_seen(g.kH * g.kW, 0);
    const WgradParams &p = L.wp;
    printf(" one launch: grid %d smem %zu groups %d x planes %d\n", L.grid, L.smem, p.n_tgrp, p.nxplane);
    CHECK(L.smem >= 1024 + (size_t)kWgradEpiBytes && L.smem <= kMaxSmem, "shared memory %zu", L.smem);
    CHECK(p.nxplane == L.nphase && p.nxplane == L.bx.nplane, "x plane count");
    for (int gi = 0; gi < p.n_tgrp; ++gi) {
        CHECK(p.grp_plane[gi] >= 0 && p.grp_plane[gi] < p.nxplane, "group %d plane", gi);
        for (int jb = p.grp_first[gi]; jb < p.grp_first[gi + 1]; ++jb) {
            printf("   grp %d (plane %d) job off %d delta %d count %d taps %d %d %d %d\n", gi, p.grp_plane[gi], p.job_off[jb],
                   p.job_delta[jb], p.job_count[jb], p.job_tapk[jb][0], p.job_tapk[jb][1], p.job_tapk[jb][2], p.job_tapk[jb][3]);
            for (int c = 0; c < p.job_count[jb]; ++c) tap_seen[p.job_tapk[jb][c]]++;
            CHECK(p.job_off[jb] + (p.job_count[jb] - 1) * p.job_delta[jb] + 128 <= p.plane_elems, "B rows");
            CHECK(p.job_col[jb] + p.job_count[jb] * 64 <= p.grp_cols[gi] && p.grp_cols[gi] <= 512, "cols");
            // every tap of the job lies in the group's phase plane: tap (kh, kw) reads x rows
            // s*oh + kh*d - pt, whose stride phase must be the plane's
            for (int c = 0; c < p.job_count[jb]; ++c) {
                const int kh = p.job_tapk[jb][c] / g.kW, kw = p.job_tapk[jb][c] % g.kW;
                const int pl = p.grp_plane[gi];
                const int rh = ((kh * g.d_h - g.pt) % g.s_h + g.s_h) % g.s_h, rw = ((kw * g.d_w - g.pl) % g.s_w + g.s_w) % g.s_w;
                const int ph = ((L.bx.roff[pl] % g.s_h) + g.s_h) % g.s_h, pw = ((L.bx.coff[pl] % g.s_w) + g.s_w) % g.s_w;
                CHECK(rh == ph && rw == pw, "tap (%d,%d) in plane %d of phase (%d,%d)", kh, kw, pl, ph, pw);
            }
        }
    }
    for (int cta = 0; cta < L.grid; ++cta) {
        int t = cta;
        const int r = t % p.cta_per_cg; t /= p.cta_per_cg;
        const int ct = t % p.n_ctile; t /= p.n_ctile;
        const int ot = t % p.n_otile;
        const int gg = t / p.n_otile;
        CHECK(gg < p.G, "cta %d group", cta);
        int gi = 0;
        while (gi + 1 < p.n_tgrp && r >= p.grp_cta0[gi + 1]) ++gi;
        const int split = r - p.grp_cta0[gi];
        const int64_t xpl = (int64_t)p.grp_plane[gi] * p.N * p.G * p.ncx;
        const int total_tiles = p.N * p.n_rowblk;
        const int tps = (total_tiles + p.grp_splits[gi] - 1) / p.grp_splits[gi];
        const int tile0 = split * tps, tile1 = std::min(total_tiles, tile0 + tps);
        const int plane_y = p.Ho * p.Wp, plane_x = p.Rx * p.Wp, th_pos = p.TH * p.Wp;
        for (int it = tile0; it < tile1; ++it) {
            const int rb = it / p.N, n = it - rb * p.N;
            const int pos0 = rb * p.TH * p.Wp;
            for (int h = 0; h < 2; ++h)
                for (int m = 0; m < 128; ++m) {
                    const int chunk = 2 * ot + h;
                    if (m < th_pos && pos0 + m < plane_y && chunk < p.ncy) {
                        const int64_t e = ((((int64_t)n * p.G + gg) * p.ncy + chunk) * plane_y + pos0 + m) * 64 + 56;
                        CHECK((size_t)(e + 8) <= yt_elems, "dy src");
                    }
                }
            for (int m = 0; m < p.plane_elems; ++m)
                if (pos0 + m < plane_x) {
                    const int64_t e = ((xpl + ((int64_t)n * p.G + gg) * p.ncx + ct) * plane_x + pos0 + m) * 64 + 56;
                    CHECK((size_t)(e + 8) <= xt_elems, "x src");
                    const int64_t lo = (int64_t)p.grp_plane[gi] * L.xplane_elems;
                    CHECK(e >= lo && (size_t)(e + 8) <= (size_t)lo + L.xplane_elems, "x within the group's phase plane");
                }
        }
        for (int jb = p.grp_first[gi]; jb < p.grp_first[gi + 1]; ++jb)
            for (int j = 0; j < p.job_count[jb]; ++j)
                for (int o = 0; o < std::min(128, p.Cgo - ot * 128); ++o) {
                    const int64_t e = (int64_t)split * ((int64_t)p.G * p.Cgo * p.Cgi * p.kHW) +
                                      ((int64_t)p.job_tapk[jb][j] * p.G * p.Cgo + gg * p.Cgo + ot * 128 + o) * p.Cgi + ct * 64 +
                                      std::min(64, p.Cgi - ct * 64) - 1;
                    CHECK((size_t)e < part_elems, "part");
                }
    }
    for (int k = 0; k < g.kH * g.kW; ++k) CHECK(tap_seen[k] == 1, "tap %d covered %d times", k, tap_seen[k]);
    printf("errors: %ld\n", errors);
    return errors ? 1 : 0;
}
