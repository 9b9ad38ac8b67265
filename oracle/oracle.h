/*
 * oracle.h -- fp64 CPU oracle for the 3-D convolution / transposed
 * convolution hot path and its fused epilogues.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or call this code.  It
 * shares nothing with the CUDA path: no headers, tables, helpers or constants.
 *
 * Every function is a plain loop nest of a definition, in fp64, on
 * contiguous NCDHW arrays (the last spatial axis fastest).  Spatial axes are
 * positional: (S0, S1, S2), S2 contiguous.  Sources are the four web pages
 * of the POPCORNBENCH transcripts, cited by page title:
 *   "Kimi-K2.6 l1_p59"  Conv3d with an asymmetric (k,k,1) kernel
 *   "Kimi-K2.6 l2_p72"  ConvTranspose3d -> BatchNorm3d -> AvgPool3d -> AvgPool3d
 *   "Kimi-K2.6 l2_p43"  Conv3d -> MaxPool3d -> logsumexp(dim=1) -> ReLU
 *   "Kimi-K2.6 l1_p77"  ConvTranspose3d with stride 2, padding 1, dilation 2
 *
 * Return value of every int function: 0 on success, -1 on an invalid
 * argument (non-positive size, indivisible groups, empty output).
 */
#ifndef TC3D_ORACLE_H
#define TC3D_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Output length of one axis of a convolution (l1_p59, output-size check of
 * the depth axis): floor((L + 2p - d(k-1) - 1)/s) + 1. Returns <= 0 if empty. */
int64_t oracle_conv_out_len(int64_t L, int k, int s, int p, int d);

/* Output length of one axis of a transposed convolution (l1_p77, output-size
 * formula): (L-1)s - 2p + d(k-1) + output_padding + 1. */
int64_t oracle_convT_out_len(int64_t L, int k, int s, int p, int d, int op);

/* Conv3d, gather form (l1_p59 direct-convolution definition with per-axis
 * stride/padding/dilation; groups as PyTorch defines them).
 * x [N,Cin,S0,S1,S2], w [Cout,Cin/G,k0,k1,k2], b [Cout] or NULL,
 * y [N,Cout,O0,O1,O2].  nthreads <= 0 means 1. */
int oracle_conv3d(const double *x, const double *w, const double *b, double *y,
                  int N, int Cin, int S0, int S1, int S2, int Cout,
                  int k0, int k1, int k2, const int stride[3], const int pad[3],
                  const int dil[3], int groups, int nthreads);

/* Same definition evaluated only at `count` flat output indices idx[i]
 * (NCDHW order of y); results in out[i]. */
int oracle_conv3d_at(const double *x, const double *w, const double *b,
                     int N, int Cin, int S0, int S1, int S2, int Cout,
                     int k0, int k1, int k2, const int stride[3], const int pad[3],
                     const int dil[3], int groups, const int64_t *idx,
                     int64_t count, double *out, int nthreads);

/* ConvTranspose3d, gather ("receive") form (l1_p77, receive-form index
 * derivation): y[n,oc,z] = b[oc] + sum_{ic in group, k} W[ic, oc', k] *
 * x[n, ic, (z + p - d k)/s] over the taps where the division is exact and the
 * quotient is in range.  w [Cin, Cout/G, k0,k1,k2]. */
int oracle_conv_transpose3d(const double *x, const double *w, const double *b,
                            double *y, int N, int Cin, int S0, int S1, int S2,
                            int Cout, int k0, int k1, int k2, const int stride[3],
                            const int pad[3], const int dil[3],
                            const int out_pad[3], int groups, int nthreads);

int oracle_conv_transpose3d_at(const double *x, const double *w, const double *b,
                               int N, int Cin, int S0, int S1, int S2, int Cout,
                               int k0, int k1, int k2, const int stride[3],
                               const int pad[3], const int dil[3],
                               const int out_pad[3], int groups,
                               const int64_t *idx, int64_t count, double *out,
                               int nthreads);

/* ConvTranspose3d, scatter form (l1_p77, scatter view): every input element
 * x[n,ic,i] times W[ic,oc',k] is added to y[n,oc,i*s - p + d*k] when that
 * index is in range.  An independent second formulation of the same result. */
int oracle_conv_transpose3d_scatter(const double *x, const double *w,
                                    const double *b, double *y, int N, int Cin,
                                    int S0, int S1, int S2, int Cout, int k0,
                                    int k1, int k2, const int stride[3],
                                    const int pad[3], const int dil[3],
                                    const int out_pad[3], int groups);

/* MaxPool3d(kernel 2, stride 2), floor mode, no padding (l2_p43 pooled-size
 * derivation).  t [N,C,L0,L1,L2] -> out [N,C,L0/2,L1/2,L2/2]. */
int oracle_maxpool3d_2(const double *t, double *out, int N, int C, int L0,
                       int L1, int L2);

/* AvgPool3d(kernel 2, stride 2), floor mode (l2_p72 pooled-size derivation). */
int oracle_avgpool3d_2(const double *t, double *out, int N, int C, int L0,
                       int L1, int L2);

/* logsumexp over the channel axis, keepdim (l2_p43 problem statement):
 * out[n,0,s] = m + log(sum_c exp(t[n,c,s] - m)), m = max_c t[n,c,s]. */
int oracle_logsumexp_channels(const double *t, double *out, int N, int C,
                              int64_t L);

/* ReLU in place: t = max(t, 0). */
void oracle_relu(double *t, int64_t n);

/* BatchNorm3d forward in training mode (l2_p72 batch-statistics discussion):
 * per channel c, mean and biased variance over (N, all spatial positions);
 * out = (t - mean) / sqrt(var + eps) * gamma[c] + beta[c].  gamma/beta may
 * be NULL (1 and 0).  mean_out / var_out (may be NULL) receive the stats. */
int oracle_batchnorm3d_train(const double *t, double *out, int N, int C,
                             int64_t L, const double *gamma, const double *beta,
                             double eps, double *mean_out, double *var_out);

/* BatchNorm3d forward in evaluation mode (the l2_p72 page's own fused
 * kernel, which read running statistics): per channel c,
 * out = (t - rmean[c]) / sqrt(rvar[c] + eps) * gamma[c] + beta[c].
 * gamma/beta may be NULL (1 and 0). */
int oracle_batchnorm3d_eval(const double *t, double *out, int N, int C,
                            int64_t L, const double *rmean, const double *rvar,
                            const double *gamma, const double *beta, double eps);

/* Composite: ConvTranspose3d(+bias) -> BatchNorm3d (running stats, eval
 * mode) -> AvgPool3d(2) -> AvgPool3d(2), each step literally, in that order.
 * y [N, Cout, P0, P1, P2] with P = floor(floor(O/2)/2). */
int oracle_convT_bneval_avgpool(const double *x, const double *w, const double *b,
                                const double *rmean, const double *rvar,
                                const double *gamma, const double *beta, double eps,
                                double *y, int N, int Cin, int S0, int S1, int S2,
                                int Cout, int k0, int k1, int k2, const int stride[3],
                                const int pad[3], const int dil[3],
                                const int out_pad[3], int groups, int nthreads);

/* Same composite at `count` flat indices of y (each pooled output from its
 * 64 transposed-conv points; no statistics are needed). */
int oracle_convT_bneval_avgpool_at(const double *x, const double *w, const double *b,
                                   const double *rmean, const double *rvar,
                                   const double *gamma, const double *beta, double eps,
                                   int N, int Cin, int S0, int S1, int S2, int Cout,
                                   int k0, int k1, int k2, const int stride[3],
                                   const int pad[3], const int dil[3],
                                   const int out_pad[3], int groups,
                                   const int64_t *idx, int64_t count, double *out,
                                   int nthreads);

/* Composite: ConvTranspose3d(+bias) -> BatchNorm3d (batch stats) ->
 * AvgPool3d(2) -> AvgPool3d(2), each step literally, in that order (l2_p72).
 * y [N, Cout, P0, P1, P2] with P = floor(floor(O/2)/2). */
int oracle_convT_bn_avgpool(const double *x, const double *w, const double *b,
                            const double *gamma, const double *beta, double eps,
                            double *y, int N, int Cin, int S0, int S1, int S2,
                            int Cout, int k0, int k1, int k2, const int stride[3],
                            const int pad[3], const int dil[3],
                            const int out_pad[3], int groups, int nthreads);

/* Same composite at `count` flat indices of y.  The batch statistics are
 * still taken over the whole transposed-conv output (streamed per (n, c)
 * slice and combined exactly); only the pooled outputs are sampled.
 * mean_out/var_out (length Cout, may be NULL) receive the statistics. */
int oracle_convT_bn_avgpool_at(const double *x, const double *w, const double *b,
                               const double *gamma, const double *beta,
                               double eps, int N, int Cin, int S0, int S1,
                               int S2, int Cout, int k0, int k1, int k2,
                               const int stride[3], const int pad[3],
                               const int dil[3], const int out_pad[3],
                               int groups, const int64_t *idx, int64_t count,
                               double *out, double *mean_out, double *var_out,
                               int nthreads);

/* Composite: Conv3d(+bias) -> MaxPool3d(2,2) -> logsumexp over channels
 * (keepdim) -> ReLU, each step literally (l2_p43).
 * y [N, 1, floor(O0/2), floor(O1/2), floor(O2/2)]. */
int oracle_conv_maxpool_lse_relu(const double *x, const double *w,
                                 const double *b, double *y, int N, int Cin,
                                 int S0, int S1, int S2, int Cout, int k0,
                                 int k1, int k2, const int stride[3],
                                 const int pad[3], const int dil[3], int groups,
                                 int nthreads);

int oracle_conv_maxpool_lse_relu_at(const double *x, const double *w,
                                    const double *b, int N, int Cin, int S0,
                                    int S1, int S2, int Cout, int k0, int k1,
                                    int k2, const int stride[3],
                                    const int pad[3], const int dil[3],
                                    int groups, const int64_t *idx,
                                    int64_t count, double *out, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
