// CPU replay of the register-blocked 3x3 stride-1 CUDA-core kernels' launch plans and index
// arithmetic for one geometry: the forward / backward-data kernel (several consecutive
// groups per block on small planes) and the weight-gradient kernel (several images staged
// at a time).  For every block and every thread it recomputes, exactly as the kernels do,
// the shared-memory writes of the staging, the shared-memory reads of the compute, and the
// global reads and writes, and checks them against the extents of the buffers.  Host code
// only: the library source is included and the device-facing helpers it calls are stubbed.
// Usage: thin3_plan_replay <14 geometry ints> <dtype: 0 fp32, 1 bf16>; exits non-zero and
// prints FAIL lines on any violation.
#include "../../bwd_gconv_fwd_gb300/csrc/direct_tiled.cu"
#include <cstdio>
#include <cstdlib>
#include <vector>
namespace gconv {
long long wait_limit() { return 1000000000LL; }
int num_sms() { return 152; }
unsigned int *device_error_word() { return nullptr; }
int forced_path() { return 0; }
int wgrad_tma_enabled() { return 1; }
void *debug_trace(size_t *b) { *b = 0; return nullptr; }
}
using namespace gconv;
static long errors = 0;
#define CHECK(cond, ...) do { if (!(cond)) { if (errors++ < 10) { printf("FAIL: " __VA_ARGS__); printf("\n"); } } } while (0)

// Staged rows of stage_rows_vec / stage_rows: every (row, column) written, as float offsets.
static void staging_writes(bool vec, int V, int nch, int RI, int CI, int CIp, int64_t dst0, int64_t dst_end,
                           const char *what)
{
    const int64_t nrows = (int64_t)nch * RI;
    if (vec) {
        const int nv = CIp / V;
        CHECK(nv * V == CIp, "%s: pitch %d not a multiple of the vector %d", what, CIp, V);
        CHECK(dst0 % 4 == 0, "%s: staged base not 16-byte aligned", what);
        for (int64_t row = 0; row < nrows; ++row) {
            const int64_t last = dst0 + row * CIp + (int64_t)(nv - 1) * V + V;   // one past the last float written
            CHECK(last <= dst_end, "%s: staged row %lld ends at %lld > %lld", what, (long long)row, (long long)last,
                  (long long)dst_end);
        }
    } else {
        for (int64_t row = 0; row < nrows; ++row)
            CHECK(dst0 + row * CIp + CI <= dst_end, "%s: staged row %lld past the buffer", what, (long long)row);
        CHECK(CI <= CIp, "%s: staged columns %d > pitch %d", what, CI, CIp);
    }
}

static void replay_conv3(const Geom &g, bool bwd, int V)
{
    Conv3Params p;
    size_t smem = 0;
    if (!plan_conv3(g, bwd, &p, &smem)) { printf("conv3 %s not served by this path\n", bwd ? "bwd" : "fwd"); return; }
    const int CO = conv3_slots(p.nout), BX = conv3_bx(p.nout);
    printf("conv3 %s: TH=%d TW=%d tq=%d CIp=%d GB=%d n_gb=%d tiles=%lld smem=%zu\n", bwd ? "bwd" : "fwd", p.TH, p.TW, p.tq,
           p.CIp, p.GB, p.n_gb, (long long)p.N * p.n_gb * p.n_th * p.n_tw, smem);
    CHECK(smem <= 96 * 1024, "conv3 shared memory %zu", smem);
    const int RI = p.TH + 2, CI = p.TW + 2, CIp = p.CIp;
    const int64_t wsz = (p.GB * p.nin * 9 * CO + 3) & ~3;
    const int64_t smem_floats = (int64_t)smem / 4;
    CHECK(wsz + (int64_t)p.GB * p.nin * RI * CIp <= smem_floats, "conv3 regions exceed the allocation");
    const int tpg = p.tq * (p.TH / 4);
    CHECK(p.GB * tpg <= kTT, "conv3: %d groups x %d threads > block", p.GB, tpg);
    const bool vec_rows = (p.IW % V) == 0;
    const int64_t plane = (int64_t)p.IH * p.IW, out_plane = (int64_t)p.OH * p.OW;
    const int64_t src_elems = (int64_t)p.N * p.in_ctot * plane, out_elems = (int64_t)p.N * p.out_ctot * out_plane;
    const int64_t w_elems = (int64_t)g.Cout * g.Cgi * 9;
    const int64_t ntiles = (int64_t)p.N * p.n_gb * p.n_th * p.n_tw;
    const bool track = out_elems <= (int64_t)1 << 24;    // exactly-once map for outputs up to 16M elements
    std::vector<int> written(track ? out_elems : 0, 0);
    for (int64_t tile = 0; tile < ntiles; ++tile) {
        int64_t b = tile;
        const int tw = b % p.n_tw; b /= p.n_tw;
        const int th = b % p.n_th; b /= p.n_th;
        const int grp0 = (int)(b % p.n_gb) * p.GB;
        const int n = (int)(b / p.n_gb);
        const int ngr = std::min(p.GB, p.G - grp0);
        CHECK(ngr >= 1, "empty group block");
        const int r0 = th * p.TH, c0 = tw * p.TW;
        // weights: ws[i] for i < ngr*nin*9*CO, from w[...] for o < nout
        CHECK((int64_t)ngr * p.nin * 9 * CO <= wsz, "conv3 weights staged past their region");
        for (int gi = 0; gi < ngr; ++gi)
            for (int ci = 0; ci < p.nin; ++ci)
                for (int tap = 0; tap < 9; ++tap)
                    for (int o = 0; o < p.nout; ++o) {
                        const int grp = grp0 + gi;
                        const int64_t idx = p.bwd ? ((int64_t)(grp * p.nin + ci) * p.w_cin_g + o) * 9 + (8 - tap)
                                                  : ((int64_t)(grp * p.nout + o) * p.w_cin_g + ci) * 9 + tap;
                        CHECK(idx >= 0 && idx < w_elems, "conv3 weight read %lld", (long long)idx);
                    }
        // input rows: nrows = ngr*nin*RI planes' rows from the group block's first channel
        const int64_t src0 = ((int64_t)n * p.in_ctot + (int64_t)grp0 * p.nin) * plane;
        const int cs = c0 + p.c_off;
        int coff = 0;
        if (vec_rows) {
            const int ca = cs >= 0 ? cs / V * V : -((-cs + V - 1) / V) * V;
            coff = cs - ca;
            staging_writes(true, V, ngr * p.nin, RI, CI, CIp, wsz, wsz + (int64_t)p.GB * p.nin * RI * CIp, "conv3 rows");
            for (int c = 0; c < ngr * p.nin; ++c)
                for (int r = 0; r < RI; ++r) {
                    const int ih = r0 + p.r_off + r;
                    if (ih < 0 || ih >= p.IH) continue;
                    for (int iw = ca; iw < ca + CIp; ++iw)
                        if (iw >= 0 && iw < p.IW) {
                            const int64_t e = src0 + c * plane + (int64_t)ih * p.IW + iw;
                            CHECK(e >= 0 && e < src_elems, "conv3 source read");
                        }
                }
        } else {
            staging_writes(false, V, ngr * p.nin, RI, CI, CIp, wsz, wsz + (int64_t)p.GB * p.nin * RI * CIp, "conv3 rows");
        }
        CHECK(coff >= 0 && coff < V, "conv3 column shift %d", coff);
        // compute and stores, per thread
        for (int t = 0; t < kTT; ++t) {
            const int gsub = t / tpg, lt = t - gsub * tpg;
            const int tx = lt % p.tq, ty = lt / p.tq;
            const int rb = 4 * ty, cb = BX * tx;
            if (!(gsub < ngr && rb < p.TH && r0 + rb < p.OH && c0 + cb < p.OW)) continue;
            const int grp = grp0 + gsub;
            for (int ci = 0; ci < p.nin; ++ci) {
                const int64_t base = wsz + (int64_t)((gsub * p.nin + ci) * RI + rb) * CIp + cb + coff;
                const int64_t last = base + 5 * CIp + BX + 1;
                CHECK(cb + coff + BX + 2 <= CIp, "conv3 window columns past the pitch");
                CHECK(last < wsz + (int64_t)(gsub * p.nin + ci + 1) * RI * CIp, "conv3 window past its plane");
                CHECK((int64_t)(gsub * p.nin + ci) * 9 * CO + 9 * CO <= wsz, "conv3 weights read past their region");
            }
            for (int o = 0; o < p.nout; ++o)
                for (int i = 0; i < 4; ++i) {
                    const int r = r0 + rb + i;
                    if (rb + i >= p.TH || r >= p.OH) break;
                    for (int j = 0; j < BX; ++j) {
                        if (c0 + cb + j >= p.OW) break;
                        const int64_t e = ((int64_t)n * p.out_ctot + (int64_t)grp * p.nout + o) * out_plane +
                                          (int64_t)r * p.OW + c0 + cb + j;
                        CHECK(e >= 0 && e < out_elems, "conv3 store");
                        if (track && e >= 0 && e < out_elems) written[e]++;
                    }
                }
        }
    }
    if (track)
        for (int64_t e = 0; e < out_elems; ++e) CHECK(written[e] == 1, "conv3 output %lld written %d times", (long long)e, written[e]);
}

static void replay_wgrad3(const Geom &g, int V)
{
    TileGeom t;
    size_t smem = 0;
    int CIpx = 0, CIpy = 0;
    if (!plan_wgrad3(g, &t, &smem, &CIpx, &CIpy)) { printf("wgrad3 not served by this path\n"); return; }
    const int IMG = std::max(1, t.IMG);
    printf("wgrad3: P=%d L=%d TH=%d TW=%d NB=%d n_nb=%d IMG=%d smem=%zu\n", t.P, t.L, t.TH, t.TW, t.NB, t.n_nb, IMG, smem);
    CHECK(smem <= 96 * 1024, "wgrad3 shared memory %zu", smem);
    CHECK(t.P * t.L <= kTT, "wgrad3 lanes");
    const int RI = t.TH + 2;
    const int64_t xsz = (int64_t)g.Cgi * RI * CIpx, dsz = (int64_t)g.Cgo * t.TH * CIpy;
    const int64_t smem_floats = (int64_t)smem / 4;
    CHECK(IMG * (xsz + dsz) <= smem_floats, "wgrad3 staged images exceed the allocation");
    CHECK((int64_t)t.P * 9 * t.L <= smem_floats, "wgrad3 reduction buffer exceeds the allocation");
    const bool xvec = (g.W % V) == 0, yvec = (g.Wo % V) == 0;
    const int nbc = t.TW / 4, nblk = (t.TH / 4) * nbc;
    const int64_t nblocks = (int64_t)g.G * t.n_th * t.n_tw * t.n_nb;
    const int64_t part_floats = nblocks * t.P * 9;
    for (int64_t blk = 0; blk < nblocks; ++blk) {
        int64_t b = blk;
        const int nb = b % t.n_nb; b /= t.n_nb;
        const int tw = b % t.n_tw; b /= t.n_tw;
        const int th = b % t.n_th; b /= t.n_th;
        const int r0 = th * t.TH, c0 = tw * t.TW;
        const int csx = c0 - g.pl;
        const int cax = xvec ? (csx >= 0 ? csx / V * V : -((-csx + V - 1) / V) * V) : csx;
        const int cay = yvec ? c0 / V * V : c0;
        const int coffx = csx - cax, coffy = c0 - cay;
        const int n1 = std::min(g.N, (nb + 1) * t.NB);
        for (int n = nb * t.NB; n < n1; n += IMG) {
            const int ni = std::min(IMG, n1 - n);
            for (int ii = 0; ii < ni; ++ii) {
                CHECK(n + ii < g.N, "wgrad3 image %d", n + ii);
                staging_writes(xvec, V, g.Cgi, RI, t.TW + 2, CIpx, ii * xsz, (ii + 1) * xsz, "wgrad3 x");
                staging_writes(yvec, V, g.Cgo, t.TH, t.TW, CIpy, IMG * xsz + ii * dsz, IMG * xsz + (ii + 1) * dsz,
                               "wgrad3 dy");
            }
            for (int q = 0; q < t.P; ++q) {
                const int o = q / g.Cgi, c = q - o * g.Cgi;
                for (int it = 0; it < ni * nblk; ++it) {
                    const int ii = it / nblk, bk = it - ii * nblk;
                    const int br = bk / nbc, bc = bk - br * nbc;
                    const int rr = 4 * br, cc = 4 * bc;
                    if (r0 + rr >= g.Ho || c0 + cc >= g.Wo) continue;
                    const int64_t xs0 = ii * xsz + (int64_t)c * RI * CIpx + coffx;
                    const int64_t ds0 = IMG * xsz + ii * dsz + (int64_t)o * t.TH * CIpy + coffy;
                    CHECK(cc + coffx + 6 <= CIpx && cc + coffy + 4 <= CIpy, "wgrad3 window columns past the pitch");
                    CHECK(xs0 + (int64_t)(rr + 5) * CIpx + cc + 5 < ii * xsz + (int64_t)(c + 1) * RI * CIpx,
                          "wgrad3 x window past its plane");
                    CHECK(ds0 + (int64_t)(rr + 3) * CIpy + cc + 3 < IMG * xsz + ii * dsz + (int64_t)(o + 1) * t.TH * CIpy,
                          "wgrad3 dy window past its plane");
                }
            }
        }
        CHECK((blk + 1) * t.P * 9 <= part_floats, "wgrad3 partial sums");
    }
}

int main(int argc, char **argv)
{
    if (argc != 16 && argc != 18) { printf("usage: thin3_plan_replay <14 or 16 geometry ints> <dtype>\n"); return 2; }
    // 14 geometry integers (one stride, one dilation) or 16 (per axis), then the dtype
    int v[16];
    const int V = atoi(argv[argc - 1]) == 1 ? 8 : 4;
    if (argc == 16) {
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
    replay_conv3(g, false, V);
    replay_conv3(g, true, V);
    replay_wgrad3(g, V);
    printf("errors: %ld\n", errors);
    return errors ? 1 : 0;
}
