/*
 * Oracle for the forward multi-channel 2-D convolution — TEST INFRASTRUCTURE.
 *
 * This file is the slow, obviously-correct reference that the CUDA path is
 * checked against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it.  It shares no code, header, table or helper with the
 * CUDA library, and the CUDA library never calls it.
 *
 * Every function works in double precision and takes its inputs already
 * widened to double from the exact bits the GPU sees (fp32, fp16 or bf16).
 *
 * What is computed (the plain definition):
 *
 *   Y[n,co,ho,wo] = sum_{ci,kh,kw} X[n,ci,ho*s+kh-p, wo*s+kw-p] * W[co,ci,kh,kw]
 *
 * with X read as zero outside [0,H) x [0,W).  Sources:
 *   - "Enabling Memory-efficient Im2win Convolution with Multi-precision
 *     Support on GPU CUDA and Tensor Cores", Sec. III-A, Eq. (1): the sum
 *     over channel, filter row and filter column, a cross-correlation
 *     (no kernel flip), written there 1-based and without stride or padding.
 *   - "Unifying Convolutions and GEMM", Sec. 1 (the naive 7-loop): the loop
 *     order n, co, ho, wo, ci, kh, kw and the ho*stride+kh indexing.
 *   - "Unifying Convolutions and GEMM", Sec. 5, and "im2col Expansion, FFT
 *     Convolution, and Winograd Transforms", im2col section: the output size
 *     H_out = (H + 2p - K_H) // s + 1 (floor) and symmetric zero padding.
 *
 * Alongside Y every direct routine returns S[n,co,ho,wo] = sum |x*w| over the
 * same terms; parity is measured as |y_gpu - Y| / S.  An optional bias
 * (oracle_add_bias, the `Y_col += bias` of "Unifying Convolutions and GEMM",
 * Sec. 6) adds b[co] to Y and |b[co]| to S.
 *
 * Parity pins (tests/test_oracle_pins.py) tie each routine to something other
 * than itself: brute force in Python, scipy's 2-D correlation, float64
 * torch.nn.functional.conv2d, closed forms (delta kernel, all-ones counts,
 * 1x1 kernel as a per-pixel matrix product, dense layer as a global-kernel
 * convolution), the worked examples printed on the pages, and invariants.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

/* Output extent along one axis, "Unifying Convolutions and GEMM" Sec. 5:
 * floor((in + 2*pad - k) / stride) + 1.  Returns 0 when no window fits. */
static int64_t out_extent(int64_t in, int64_t k, int64_t s, int64_t p)
{
    int64_t span = in + 2 * p - k;
    if (span < 0 || s < 1) return 0;
    return span / s + 1;
}

int oracle_out_dims(int H, int W, int Kh, int Kw, int s, int p, int *Ho, int *Wo)
{
    *Ho = (int)out_extent(H, Kh, s, p);
    *Wo = (int)out_extent(W, Kw, s, p);
    return (*Ho > 0 && *Wo > 0) ? 0 : -1;
}

/* One output element by the definition: the three inner loops of the 7-loop
 * (ci, kh, kw), with out-of-image taps contributing nothing. */
static void one_output(const double *X, const double *Wt,
                       int64_t Ci, int64_t H, int64_t W, int64_t Kh, int64_t Kw,
                       int64_t s, int64_t p,
                       int64_t n, int64_t co, int64_t ho, int64_t wo,
                       double *y_out, double *s_out)
{
    double acc = 0.0, sabs = 0.0;
    for (int64_t ci = 0; ci < Ci; ++ci) {
        const double *xc = X + ((n * Ci + ci) * H) * W;
        const double *wc = Wt + ((co * Ci + ci) * Kh) * Kw;
        for (int64_t kh = 0; kh < Kh; ++kh) {
            int64_t y = ho * s + kh - p;
            if (y < 0 || y >= H) continue;
            for (int64_t kw = 0; kw < Kw; ++kw) {
                int64_t x = wo * s + kw - p;
                if (x < 0 || x >= W) continue;
                double t = xc[y * W + x] * wc[kh * Kw + kw];
                acc += t;
                sabs += fabs(t);
            }
        }
    }
    *y_out = acc;
    if (s_out) *s_out = sabs;
}

/* The 7-loop over the slice n in [n0,n1), co in [co0,co1).  Y and S are the
 * full NCHW output arrays; only the slice is written.  S may be NULL. */
int oracle_conv2d_direct_slice(const double *X, const double *Wt, double *Y, double *S,
                               int N, int Ci, int H, int W, int Co, int Kh, int Kw,
                               int s, int p, int n0, int n1, int co0, int co1)
{
    int Ho, Wo;
    if (N < 0 || Ci < 1 || Co < 1 || Kh < 1 || Kw < 1 || s < 1 || p < 0) return -1;
    if (oracle_out_dims(H, W, Kh, Kw, s, p, &Ho, &Wo) != 0) return -1;
    for (int64_t n = n0; n < n1; ++n)
        for (int64_t co = co0; co < co1; ++co)
            for (int64_t ho = 0; ho < Ho; ++ho)
                for (int64_t wo = 0; wo < Wo; ++wo) {
                    int64_t o = ((n * Co + co) * Ho + ho) * Wo + wo;
                    one_output(X, Wt, Ci, H, W, Kh, Kw, s, p, n, co, ho, wo,
                               &Y[o], S ? &S[o] : NULL);
                }
    return 0;
}

int oracle_conv2d_direct(const double *X, const double *Wt, double *Y, double *S,
                         int N, int Ci, int H, int W, int Co, int Kh, int Kw, int s, int p)
{
    return oracle_conv2d_direct_slice(X, Wt, Y, S, N, Ci, H, W, Co, Kh, Kw, s, p,
                                      0, N, 0, Co);
}

/* Selected outputs only: idx[i] is the flat NCHW index of output i.  Used to
 * check full-size runs on a sample the oracle can afford. */
int oracle_conv2d_points(const double *X, const double *Wt, const int64_t *idx, int64_t npts,
                         double *Y, double *S,
                         int N, int Ci, int H, int W, int Co, int Kh, int Kw, int s, int p)
{
    int Ho, Wo;
    if (oracle_out_dims(H, W, Kh, Kw, s, p, &Ho, &Wo) != 0) return -1;
    int64_t total = (int64_t)N * Co * Ho * Wo;
    for (int64_t i = 0; i < npts; ++i) {
        int64_t o = idx[i];
        if (o < 0 || o >= total) return -2;
        int64_t wo = o % Wo, r = o / Wo;
        int64_t ho = r % Ho;  r /= Ho;
        int64_t co = r % Co, n = r / Co;
        one_output(X, Wt, Ci, H, W, Kh, Kw, s, p, n, co, ho, wo, &Y[i], S ? &S[i] : NULL);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Independent path: im2col expansion followed by a naive matrix product.
 *
 * im2col ("im2col Expansion, FFT Convolution, and Winograd Transforms",
 * im2col section): for one sample, a (Ci*Kh*Kw) x (Ho*Wo) matrix whose row
 * (ci,kh,kw) holds, for every output cell, the zero-padded input element that
 * tap sees.  GEMM ("Unifying Convolutions and GEMM", Sec. 3): with W viewed
 * as a Co x (Ci*Kh*Kw) matrix, Y_n = W_row * cols_n.
 * ------------------------------------------------------------------------- */
int oracle_im2col(const double *Xn, double *cols, int Ci, int H, int W,
                  int Kh, int Kw, int s, int p)
{
    int Ho, Wo;
    if (oracle_out_dims(H, W, Kh, Kw, s, p, &Ho, &Wo) != 0) return -1;
    int64_t L = (int64_t)Ho * Wo;
    int64_t row = 0;
    for (int64_t ci = 0; ci < Ci; ++ci)
        for (int64_t kh = 0; kh < Kh; ++kh)
            for (int64_t kw = 0; kw < Kw; ++kw, ++row)
                for (int64_t ho = 0; ho < Ho; ++ho)
                    for (int64_t wo = 0; wo < Wo; ++wo) {
                        int64_t y = ho * s + kh - p, x = wo * s + kw - p;
                        double v = 0.0;
                        if (y >= 0 && y < H && x >= 0 && x < W)
                            v = Xn[((ci * H) + y) * W + x];
                        cols[row * L + ho * Wo + wo] = v;
                    }
    return 0;
}

/* C[M][N] = A[M][K] * B[K][N], all row-major, triple loop. */
void oracle_gemm_naive(const double *A, const double *B, double *C, int M, int N, int K)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += A[i * (int64_t)K + k] * B[k * (int64_t)N + j];
            C[i * (int64_t)N + j] = acc;
        }
}

/* Whole convolution through im2col + GEMM; cols is caller scratch of
 * Ci*Kh*Kw*Ho*Wo doubles. */
int oracle_conv2d_im2col(const double *X, const double *Wt, double *Y, double *cols,
                         int N, int Ci, int H, int W, int Co, int Kh, int Kw, int s, int p)
{
    int Ho, Wo;
    if (oracle_out_dims(H, W, Kh, Kw, s, p, &Ho, &Wo) != 0) return -1;
    int64_t K = (int64_t)Ci * Kh * Kw, L = (int64_t)Ho * Wo;
    for (int64_t n = 0; n < N; ++n) {
        oracle_im2col(X + n * (int64_t)Ci * H * W, cols, Ci, H, W, Kh, Kw, s, p);
        oracle_gemm_naive(Wt, cols, Y + n * (int64_t)Co * L, Co, (int)L, (int)K);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * im2win, "Enabling Memory-efficient Im2win Convolution ...", Sec. III-B,
 * Eq. (2) and Sec. III-C, Eq. (3), translated to 0-based indices and extended
 * with symmetric zero padding.
 *
 * Transform (Eq. 2): for output row m of channel r of sample i, the strip
 *     Xw[i][r][m][k*Kh + u] = Xpad[i][r][m*s + u][k],   k in [0,Wp), u in [0,Kh)
 * where Xpad is X surrounded by p zeros on every side and Wp = W + 2p.  Each
 * input column k contributes its Kh vertically adjacent elements contiguously.
 *
 * Convolution (Eq. 3): output (i,j,m,n) sums, over r, u, v,
 *     Xw[i][r][m][(n*s + v)*Kh + u] * F[j][r][u][v].
 * The printed index multiplies by the filter width; the strip of Eq. (2)
 * advances Kh elements per input column, so the filter height is the factor
 * that makes Eq. (3) agree with Eq. (1).  The two readings coincide for square
 * filters; the tests use non-square filters to tell them apart.
 * ------------------------------------------------------------------------- */
int oracle_im2win_transform(const double *X, double *Xw, int N, int Ci, int H, int W,
                            int Kh, int Kw, int s, int p)
{
    int Ho, Wo;
    if (oracle_out_dims(H, W, Kh, Kw, s, p, &Ho, &Wo) != 0) return -1;
    int64_t Wp = (int64_t)W + 2 * p, L = Wp * Kh;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t ci = 0; ci < Ci; ++ci)
            for (int64_t m = 0; m < Ho; ++m) {
                double *strip = Xw + ((n * Ci + ci) * Ho + m) * L;
                for (int64_t k = 0; k < Wp; ++k)
                    for (int64_t u = 0; u < Kh; ++u) {
                        int64_t y = m * s + u - p, x = k - p;
                        double v = 0.0;
                        if (y >= 0 && y < H && x >= 0 && x < W)
                            v = X[((n * Ci + ci) * H + y) * W + x];
                        strip[k * Kh + u] = v;
                    }
            }
    return 0;
}

int oracle_im2win_conv(const double *Xw, const double *Wt, double *Y,
                       int N, int Ci, int H, int W, int Co, int Kh, int Kw, int s, int p)
{
    int Ho, Wo;
    if (oracle_out_dims(H, W, Kh, Kw, s, p, &Ho, &Wo) != 0) return -1;
    int64_t Wp = (int64_t)W + 2 * p, L = Wp * Kh;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t co = 0; co < Co; ++co)
            for (int64_t m = 0; m < Ho; ++m)
                for (int64_t q = 0; q < Wo; ++q) {
                    double acc = 0.0;
                    for (int64_t ci = 0; ci < Ci; ++ci) {
                        const double *strip = Xw + ((n * Ci + ci) * Ho + m) * L;
                        const double *f = Wt + (co * Ci + ci) * (int64_t)Kh * Kw;
                        for (int64_t u = 0; u < Kh; ++u)
                            for (int64_t v = 0; v < Kw; ++v)
                                acc += strip[(q * s + v) * Kh + u] * f[u * Kw + v];
                    }
                    Y[((n * Co + co) * Ho + m) * Wo + q] = acc;
                }
    return 0;
}

/* Bias of the PyTorch listing of "Unifying Convolutions and GEMM", Sec. 6
 * (manual_im2col_conv(x, weights, bias, ...), `Y_col += bias`): one value per
 * output channel, added to every output of that channel after the sum:
 *
 *   Y[n,co,ho,wo] += b[co],   S[n,co,ho,wo] += |b[co]|
 *
 * so that the parity measure |y - Y| / S also covers the bias term.  Y and S
 * are whole NCHW outputs of N x Co x Ho x Wo; S may be NULL. */
int oracle_add_bias(double *Y, double *S, const double *b, int N, int Co, int Ho, int Wo)
{
    if (N < 0 || Co < 1 || Ho < 1 || Wo < 1) return -1;
    const int64_t plane = (int64_t)Ho * Wo;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t co = 0; co < Co; ++co) {
            double *y = Y + (n * Co + co) * plane;
            double *sa = S ? S + (n * Co + co) * plane : NULL;
            for (int64_t i = 0; i < plane; ++i) {
                y[i] += b[co];
                if (sa) sa[i] += fabs(b[co]);
            }
        }
    return 0;
}
