/* CPython-API binding of the C ABI's compute calls (include/tn_gemm.h).
 *
 * Argument marshalling only, with the C ABI's names and argument order: sizes
 * and leading dimensions are Python ints, pointers are ints (device or host
 * addresses) or None for NULL, scales are floats, and each call returns the
 * C ABI's gemm_status_t as an int.  Every call goes straight to the C ABI
 * function of libdense_gemm_tn.so.
 *
 * Why it exists: a ctypes call with ten arguments costs about 1.5 us of host
 * time on the GPU machine's cores, as much as a whole small GEMM on the GPU; a
 * METH_FASTCALL function converts the same arguments in a fraction of that.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

#include "tn_gemm.h"

/* Reads args[i] as a 64-bit int; returns 0 and sets an exception on failure. */
static int arg_i64(PyObject *const *args, Py_ssize_t i, int64_t *out)
{
    long long v = PyLong_AsLongLong(args[i]);
    if (v == -1 && PyErr_Occurred()) return 0;
    *out = (int64_t)v;
    return 1;
}

static int arg_int(PyObject *const *args, Py_ssize_t i, int *out)
{
    long v = PyLong_AsLong(args[i]);
    if (v == -1 && PyErr_Occurred()) return 0;
    if (v < INT32_MIN || v > INT32_MAX) {
        PyErr_SetString(PyExc_OverflowError, "argument does not fit a C int");
        return 0;
    }
    *out = (int)v;
    return 1;
}

/* A pointer: None -> NULL, else a non-negative int address. */
static int arg_ptr(PyObject *const *args, Py_ssize_t i, void **out)
{
    if (args[i] == Py_None) {
        *out = NULL;
        return 1;
    }
    void *p = PyLong_AsVoidPtr(args[i]);
    if (p == NULL && PyErr_Occurred()) return 0;
    *out = p;
    return 1;
}

static int arg_float(PyObject *const *args, Py_ssize_t i, float *out)
{
    double v = PyFloat_AsDouble(args[i]);
    if (v == -1.0 && PyErr_Occurred()) return 0;
    *out = (float)v;
    return 1;
}

static int check_nargs(const char *name, Py_ssize_t nargs, Py_ssize_t want)
{
    if (nargs == want) return 1;
    PyErr_Format(PyExc_TypeError, "%s takes %zd arguments (%zd given)", name, want, nargs);
    return 0;
}

/* The ten-argument form shared by gemm_f16_tn and gemm_f16_tn_noalloc:
 * (M, N, K, A, lda, B, ldb, C, ldc, stream). */
typedef gemm_status_t (*f16_fn)(int64_t, int64_t, int64_t, const void *, int64_t, const void *, int64_t, void *,
                                int64_t, void *);

static PyObject *call_f16(const char *name, f16_fn fn, PyObject *const *args, Py_ssize_t nargs)
{
    int64_t M, N, K, lda, ldb, ldc;
    void *A, *B, *C, *stream;
    if (!check_nargs(name, nargs, 10) || !arg_i64(args, 0, &M) || !arg_i64(args, 1, &N) || !arg_i64(args, 2, &K) ||
        !arg_ptr(args, 3, &A) || !arg_i64(args, 4, &lda) || !arg_ptr(args, 5, &B) || !arg_i64(args, 6, &ldb) ||
        !arg_ptr(args, 7, &C) || !arg_i64(args, 8, &ldc) || !arg_ptr(args, 9, &stream))
        return NULL;
    return PyLong_FromLong((long)fn(M, N, K, A, lda, B, ldb, C, ldc, stream));
}

static PyObject *py_gemm_f16_tn(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    return call_f16("gemm_f16_tn", gemm_f16_tn, args, nargs);
}

static PyObject *py_gemm_f16_tn_noalloc(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    return call_f16("gemm_f16_tn_noalloc", gemm_f16_tn_noalloc, args, nargs);
}

/* (M, N, K, A, lda, B, ldb, C, ldc, scale_a, scale_b, stream) */
static PyObject *py_gemm_f8e4m3_tn(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    int64_t M, N, K, lda, ldb, ldc;
    void *A, *B, *C, *stream;
    float sa, sb;
    if (!check_nargs("gemm_f8e4m3_tn", nargs, 12) || !arg_i64(args, 0, &M) || !arg_i64(args, 1, &N) ||
        !arg_i64(args, 2, &K) || !arg_ptr(args, 3, &A) || !arg_i64(args, 4, &lda) || !arg_ptr(args, 5, &B) ||
        !arg_i64(args, 6, &ldb) || !arg_ptr(args, 7, &C) || !arg_i64(args, 8, &ldc) || !arg_float(args, 9, &sa) ||
        !arg_float(args, 10, &sb) || !arg_ptr(args, 11, &stream))
        return NULL;
    return PyLong_FromLong((long)gemm_f8e4m3_tn(M, N, K, A, lda, B, ldb, C, ldc, sa, sb, stream));
}

/* (M, N, K, A, lda, B, ldb, C, ldc, scale_a_ptr, scale_b_ptr, stream) */
static PyObject *py_gemm_f8e4m3_tn_dscale(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    int64_t M, N, K, lda, ldb, ldc;
    void *A, *B, *C, *sa, *sb, *stream;
    if (!check_nargs("gemm_f8e4m3_tn_dscale", nargs, 12) || !arg_i64(args, 0, &M) || !arg_i64(args, 1, &N) ||
        !arg_i64(args, 2, &K) || !arg_ptr(args, 3, &A) || !arg_i64(args, 4, &lda) || !arg_ptr(args, 5, &B) ||
        !arg_i64(args, 6, &ldb) || !arg_ptr(args, 7, &C) || !arg_i64(args, 8, &ldc) || !arg_ptr(args, 9, &sa) ||
        !arg_ptr(args, 10, &sb) || !arg_ptr(args, 11, &stream))
        return NULL;
    return PyLong_FromLong(
        (long)gemm_f8e4m3_tn_dscale(M, N, K, A, lda, B, ldb, C, ldc, (const float *)sa, (const float *)sb, stream));
}

/* (M, N, K, A, lda, B, ldb, C, ldc, scale, row_max, row_sum, stream) */
static PyObject *py_gemm_f16_tn_softmax_stats(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    int64_t M, N, K, lda, ldb, ldc;
    void *A, *B, *C, *mx, *sm, *stream;
    float scale;
    if (!check_nargs("gemm_f16_tn_softmax_stats", nargs, 13) || !arg_i64(args, 0, &M) || !arg_i64(args, 1, &N) ||
        !arg_i64(args, 2, &K) || !arg_ptr(args, 3, &A) || !arg_i64(args, 4, &lda) || !arg_ptr(args, 5, &B) ||
        !arg_i64(args, 6, &ldb) || !arg_ptr(args, 7, &C) || !arg_i64(args, 8, &ldc) ||
        !arg_float(args, 9, &scale) || !arg_ptr(args, 10, &mx) || !arg_ptr(args, 11, &sm) ||
        !arg_ptr(args, 12, &stream))
        return NULL;
    return PyLong_FromLong((long)gemm_f16_tn_softmax_stats(M, N, K, A, lda, B, ldb, C, ldc, scale, (float *)mx,
                                                           (float *)sm, stream));
}

/* (x, dtype, rows, cols, ldx, q, ldq, scale_out, stream) */
static PyObject *py_gemm_quantize_e4m3(PyObject *self, PyObject *const *args, Py_ssize_t nargs)
{
    (void)self;
    void *x, *q, *scale, *stream;
    int dtype;
    int64_t rows, cols, ldx, ldq;
    if (!check_nargs("gemm_quantize_e4m3", nargs, 9) || !arg_ptr(args, 0, &x) || !arg_int(args, 1, &dtype) ||
        !arg_i64(args, 2, &rows) || !arg_i64(args, 3, &cols) || !arg_i64(args, 4, &ldx) || !arg_ptr(args, 5, &q) ||
        !arg_i64(args, 6, &ldq) || !arg_ptr(args, 7, &scale) || !arg_ptr(args, 8, &stream))
        return NULL;
    return PyLong_FromLong(
        (long)gemm_quantize_e4m3(x, dtype, rows, cols, ldx, q, ldq, (float *)scale, stream));
}

static PyMethodDef methods[] = {
    {"gemm_f16_tn", (PyCFunction)(void (*)(void))py_gemm_f16_tn, METH_FASTCALL,
     "gemm_f16_tn(M, N, K, A, lda, B, ldb, C, ldc, stream) -> status"},
    {"gemm_f16_tn_noalloc", (PyCFunction)(void (*)(void))py_gemm_f16_tn_noalloc, METH_FASTCALL,
     "gemm_f16_tn_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream) -> status"},
    {"gemm_f8e4m3_tn", (PyCFunction)(void (*)(void))py_gemm_f8e4m3_tn, METH_FASTCALL,
     "gemm_f8e4m3_tn(M, N, K, A, lda, B, ldb, C, ldc, scale_a, scale_b, stream) -> status"},
    {"gemm_f8e4m3_tn_dscale", (PyCFunction)(void (*)(void))py_gemm_f8e4m3_tn_dscale, METH_FASTCALL,
     "gemm_f8e4m3_tn_dscale(M, N, K, A, lda, B, ldb, C, ldc, scale_a_ptr, scale_b_ptr, stream) -> status"},
    {"gemm_f16_tn_softmax_stats", (PyCFunction)(void (*)(void))py_gemm_f16_tn_softmax_stats, METH_FASTCALL,
     "gemm_f16_tn_softmax_stats(M, N, K, A, lda, B, ldb, C, ldc, scale, row_max, row_sum, stream) -> status"},
    {"gemm_quantize_e4m3", (PyCFunction)(void (*)(void))py_gemm_quantize_e4m3, METH_FASTCALL,
     "gemm_quantize_e4m3(x, dtype, rows, cols, ldx, q, ldq, scale_out, stream) -> status"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_tn_fast",
                                    "CPython-API binding of the dense TN GEMM C ABI's compute calls.", -1, methods};

PyMODINIT_FUNC PyInit__tn_fast(void) { return PyModule_Create(&module); }
