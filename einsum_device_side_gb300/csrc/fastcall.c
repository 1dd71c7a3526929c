/*
 * fastcall.c -- CPython binding of the hot entry points of include/tropical.h.
 *
 * Argument marshalling only: each function takes plain Python integers
 * (device addresses, extents, strides, dtype and semiring codes, the stream
 * handle) and tuples of them, fills the C descriptors and calls the C ABI,
 * returning its status code.  It exists because a ctypes call converting
 * twenty arguments costs about 2 us of host time per call, more than the
 * library's own planning; the vectorcall convention (METH_FASTCALL) used here
 * passes the arguments without building a tuple.  No torch type crosses it.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <string.h>

#include "tropical.h"

/* a Python int (or None = 0) as a pointer-sized integer */
static int as_ptr(PyObject* o, void** out)
{
    if (o == Py_None) {
        *out = NULL;
        return 0;
    }
    *out = PyLong_AsVoidPtr(o);
    return (*out == NULL && PyErr_Occurred()) ? -1 : 0;
}

static int as_i64(PyObject* o, int64_t* out)
{
    *out = (int64_t)PyLong_AsLongLong(o);
    return (*out == -1 && PyErr_Occurred()) ? -1 : 0;
}

/* descriptor from (address, dtype code, shape tuple, stride tuple) */
static int fill_tensor(trop_tensor* t, PyObject* ptr, PyObject* dtype, PyObject* shape, PyObject* stride)
{
    if (!PyTuple_Check(shape) || !PyTuple_Check(stride)) {
        PyErr_SetString(PyExc_TypeError, "shape and stride must be tuples");
        return -1;
    }
    const Py_ssize_t n = PyTuple_GET_SIZE(shape);
    if (n > TROP_MAX_RANK || PyTuple_GET_SIZE(stride) != n) {
        PyErr_SetString(PyExc_ValueError, "rank above 32 or shape/stride lengths differ");
        return -1;
    }
    if (as_ptr(ptr, &t->data) < 0) return -1;
    const long dt = PyLong_AsLong(dtype);
    if (dt == -1 && PyErr_Occurred()) return -1;
    t->dtype = (int32_t)dt;
    t->rank = (int32_t)n;
    for (Py_ssize_t i = 0; i < n; ++i) {
        if (as_i64(PyTuple_GET_ITEM(shape, i), &t->shape[i]) < 0) return -1;
        if (as_i64(PyTuple_GET_ITEM(stride, i), &t->stride[i]) < 0) return -1;
    }
    return 0;
}

static int check_nargs(Py_ssize_t nargs, Py_ssize_t want, const char* name)
{
    if (nargs == want) return 0;
    PyErr_Format(PyExc_TypeError, "%s takes %zd arguments (%zd given)", name, want, nargs);
    return -1;
}

/* Every tensor is passed as four arguments: address (int or None), dtype code, shape tuple,
 * stride tuple (elements). */

/* permute_trace(in x4, spec: bytes, semiring, out x4, argmax_ptr, stream, no_alloc) -> status */
static PyObject* fc_permute_trace(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    if (check_nargs(nargs, 13, "permute_trace") < 0) return NULL;
    trop_tensor in, out;
    void *argmax, *stream;
    if (fill_tensor(&in, a[0], a[1], a[2], a[3]) < 0 || fill_tensor(&out, a[6], a[7], a[8], a[9]) < 0 ||
        as_ptr(a[10], &argmax) < 0 || as_ptr(a[11], &stream) < 0)
        return NULL;
    const char* spec = PyBytes_AsString(a[4]);
    const long sr = PyLong_AsLong(a[5]);
    const int no_alloc = PyObject_IsTrue(a[12]);
    if (!spec || (sr == -1 && PyErr_Occurred()) || no_alloc < 0) return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = no_alloc ? tropical_permute_trace_noalloc(&in, spec, (int)sr, &out, (int32_t*)argmax, stream)
                  : tropical_permute_trace(&in, spec, (int)sr, &out, (int32_t*)argmax, stream);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

/* permute_pair(val_in x4, arg_in x4, spec: bytes, val_out x4, arg_out x4, stream) -> status */
static PyObject* fc_permute_pair(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    if (check_nargs(nargs, 18, "permute_pair") < 0) return NULL;
    trop_tensor vi, ai, vo, ao;
    void* stream;
    if (fill_tensor(&vi, a[0], a[1], a[2], a[3]) < 0 || fill_tensor(&ai, a[4], a[5], a[6], a[7]) < 0 ||
        fill_tensor(&vo, a[9], a[10], a[11], a[12]) < 0 || fill_tensor(&ao, a[13], a[14], a[15], a[16]) < 0 ||
        as_ptr(a[17], &stream) < 0)
        return NULL;
    const char* spec = PyBytes_AsString(a[8]);
    if (!spec) return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = tropical_permute_pair(&vi, &ai, spec, &vo, &ao, stream);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

/* gemm(semiring, dtype, batch, M, N, K, A, sAb, sAm, sAk, B, sBb, sBk, sBn, C, sCb, sCm, sCn,
 *      argmax, stream): the twenty arguments of tropical_gemm_strided_batched_argmax */
static PyObject* fc_gemm(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    if (check_nargs(nargs, 20, "gemm") < 0) return NULL;
    int64_t v[20];
    void* p[20];
    for (int i = 0; i < 20; ++i) {
        const int is_ptr = i == 6 || i == 10 || i == 14 || i == 18 || i == 19;
        if (is_ptr ? as_ptr(a[i], &p[i]) < 0 : as_i64(a[i], &v[i]) < 0) return NULL;
    }
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = tropical_gemm_strided_batched_argmax((int)v[0], (int)v[1], v[2], v[3], v[4], v[5], p[6], v[7], v[8], v[9],
                                              p[10], v[11], v[12], v[13], p[14], v[15], v[16], v[17],
                                              (int32_t*)p[18], p[19]);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

/* einsum(spec: bytes, A x4, B x4, semiring, out x4, argmax_ptr, stream) -> status */
static PyObject* fc_einsum(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    if (check_nargs(nargs, 16, "einsum") < 0) return NULL;
    trop_tensor A, B, out;
    void *argmax, *stream;
    if (fill_tensor(&A, a[1], a[2], a[3], a[4]) < 0 || fill_tensor(&B, a[5], a[6], a[7], a[8]) < 0 ||
        fill_tensor(&out, a[10], a[11], a[12], a[13]) < 0 || as_ptr(a[14], &argmax) < 0 ||
        as_ptr(a[15], &stream) < 0)
        return NULL;
    const char* spec = PyBytes_AsString(a[0]);
    const long sr = PyLong_AsLong(a[9]);
    if (!spec || (sr == -1 && PyErr_Occurred())) return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = tropical_einsum_pairwise(spec, &A, &B, (int)sr, &out, (int32_t*)argmax, stream);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

static PyObject* fc_last_error(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    (void)a;
    if (check_nargs(nargs, 0, "last_error") < 0) return NULL;
    return PyUnicode_DecodeUTF8(tropical_last_error(), (Py_ssize_t)strlen(tropical_last_error()), "replace");
}

static PyMethodDef methods[] = {
    {"permute_trace", (PyCFunction)(void (*)(void))fc_permute_trace, METH_FASTCALL, "tropical_permute_trace"},
    {"permute_pair", (PyCFunction)(void (*)(void))fc_permute_pair, METH_FASTCALL, "tropical_permute_pair"},
    {"gemm", (PyCFunction)(void (*)(void))fc_gemm, METH_FASTCALL, "tropical_gemm_strided_batched_argmax"},
    {"einsum", (PyCFunction)(void (*)(void))fc_einsum, METH_FASTCALL, "tropical_einsum_pairwise"},
    {"last_error", (PyCFunction)(void (*)(void))fc_last_error, METH_FASTCALL, "tropical_last_error"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_fastcall", "hot entry points of the C ABI", -1,
                                    methods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastcall(void) { return PyModule_Create(&module); }
