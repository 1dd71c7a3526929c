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

/* ---- tensor-taking variants: the same calls, reading each tensor's data_ptr(), dtype, shape and
 * stride() through the C API (the tensors are treated as plain Python objects with those
 * attributes), so the Python wrapper does no per-argument work.  set_torch_handles() gives the
 * dtype objects (matched by identity: float32, int32, int64, float64 -> the trop_dtype codes)
 * and the function returning a device's current raw stream. */
static PyObject* g_dtype_obj[4];
static PyObject* g_raw_stream;
static PyObject *s_data_ptr, *s_shape, *s_stride, *s_dtype, *s_get_device, *s_cuda_stream;

static PyObject* fc_set_torch_handles(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    if (check_nargs(nargs, 5, "set_torch_handles") < 0) return NULL;
    for (int i = 0; i < 4; ++i) {
        Py_XDECREF(g_dtype_obj[i]);
        Py_INCREF(a[i]);
        g_dtype_obj[i] = a[i];
    }
    Py_XDECREF(g_raw_stream);
    Py_INCREF(a[4]);
    g_raw_stream = a[4];
    Py_RETURN_NONE;
}

static int obj_tensor(trop_tensor* t, PyObject* obj)
{
    PyObject* p = PyObject_CallMethodNoArgs(obj, s_data_ptr);
    if (!p) return -1;
    const int bad = as_ptr(p, &t->data) < 0;
    Py_DECREF(p);
    if (bad) return -1;
    PyObject* dt = PyObject_GetAttr(obj, s_dtype);
    if (!dt) return -1;
    t->dtype = -1;  /* unknown dtypes reach the C ABI as -1, which it refuses */
    for (int i = 0; i < 4; ++i)
        if (dt == g_dtype_obj[i]) t->dtype = i;
    Py_DECREF(dt);
    PyObject* shape = PyObject_GetAttr(obj, s_shape);
    if (!shape) return -1;
    PyObject* stride = PyObject_CallMethodNoArgs(obj, s_stride);
    if (!stride) {
        Py_DECREF(shape);
        return -1;
    }
    int rc = 0;
    const Py_ssize_t n = PyTuple_Check(shape) && PyTuple_Check(stride) ? PyTuple_GET_SIZE(shape) : -1;
    if (n < 0 || n > TROP_MAX_RANK || PyTuple_GET_SIZE(stride) != n) {
        PyErr_SetString(PyExc_ValueError, "tensor rank above 32 or unreadable shape/stride");
        rc = -1;
    } else {
        t->rank = (int32_t)n;
        for (Py_ssize_t i = 0; i < n && rc == 0; ++i)
            if (as_i64(PyTuple_GET_ITEM(shape, i), &t->shape[i]) < 0 || as_i64(PyTuple_GET_ITEM(stride, i), &t->stride[i]) < 0)
                rc = -1;
    }
    Py_DECREF(shape);
    Py_DECREF(stride);
    return rc;
}

/* the stream handle: stream.cuda_stream, or the current raw stream of obj's device */
static int obj_stream(PyObject* stream, PyObject* obj, void** out)
{
    PyObject* h;
    if (stream != Py_None) {
        h = PyObject_GetAttr(stream, s_cuda_stream);
    } else {
        if (!g_raw_stream) {
            PyErr_SetString(PyExc_RuntimeError, "set_torch_handles was not called");
            return -1;
        }
        PyObject* dev = PyObject_CallMethodNoArgs(obj, s_get_device);
        if (!dev) return -1;
        h = PyObject_CallOneArg(g_raw_stream, dev);
        Py_DECREF(dev);
    }
    if (!h) return -1;
    const int rc = as_ptr(h, out);
    Py_DECREF(h);
    return rc;
}

static int obj_semiring(PyObject* o, long* sr)
{
    if (PyUnicode_Check(o)) {
        *sr = PyUnicode_CompareWithASCIIString(o, "maxplus") == 0    ? 0
              : PyUnicode_CompareWithASCIIString(o, "minplus") == 0  ? 1
              : PyUnicode_CompareWithASCIIString(o, "maxtimes") == 0 ? 2
                                                                      : -1;
        if (*sr < 0) {
            PyErr_SetString(PyExc_KeyError, "semiring must be 'maxplus', 'minplus' or 'maxtimes'");
            return -1;
        }
        return 0;
    }
    *sr = PyLong_AsLong(o);
    return (*sr == -1 && PyErr_Occurred()) ? -1 : 0;
}

/* permute_trace_t(x, spec: str, semiring, out, argmax tensor or None, stream or None, no_alloc) */
static PyObject* fc_permute_trace_t(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    if (check_nargs(nargs, 7, "permute_trace_t") < 0) return NULL;
    trop_tensor in, out;
    void *argmax = NULL, *stream;
    long sr;
    if (obj_tensor(&in, a[0]) < 0 || obj_tensor(&out, a[3]) < 0 || obj_semiring(a[2], &sr) < 0 ||
        obj_stream(a[5], a[0], &stream) < 0)
        return NULL;
    if (a[4] != Py_None) {
        PyObject* p = PyObject_CallMethodNoArgs(a[4], s_data_ptr);
        if (!p) return NULL;
        const int bad = as_ptr(p, &argmax) < 0;
        Py_DECREF(p);
        if (bad) return NULL;
    }
    const char* spec = PyUnicode_AsUTF8(a[1]);
    const int no_alloc = PyObject_IsTrue(a[6]);
    if (!spec || no_alloc < 0) return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = no_alloc ? tropical_permute_trace_noalloc(&in, spec, (int)sr, &out, (int32_t*)argmax, stream)
                  : tropical_permute_trace(&in, spec, (int)sr, &out, (int32_t*)argmax, stream);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(rc);
}

/* permute_pair_t(val, arg, spec: str, out_val, out_arg, stream or None) */
static PyObject* fc_permute_pair_t(PyObject* self, PyObject* const* a, Py_ssize_t nargs)
{
    (void)self;
    if (check_nargs(nargs, 6, "permute_pair_t") < 0) return NULL;
    trop_tensor vi, ai, vo, ao;
    void* stream;
    if (obj_tensor(&vi, a[0]) < 0 || obj_tensor(&ai, a[1]) < 0 || obj_tensor(&vo, a[3]) < 0 ||
        obj_tensor(&ao, a[4]) < 0 || obj_stream(a[5], a[0], &stream) < 0)
        return NULL;
    const char* spec = PyUnicode_AsUTF8(a[2]);
    if (!spec) return NULL;
    int rc;
    Py_BEGIN_ALLOW_THREADS
    rc = tropical_permute_pair(&vi, &ai, spec, &vo, &ao, stream);
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
    {"set_torch_handles", (PyCFunction)(void (*)(void))fc_set_torch_handles, METH_FASTCALL,
     "dtype objects (float32, int32, int64, float64) and the current-raw-stream function"},
    {"permute_trace_t", (PyCFunction)(void (*)(void))fc_permute_trace_t, METH_FASTCALL,
     "tropical_permute_trace on tensor objects"},
    {"permute_pair_t", (PyCFunction)(void (*)(void))fc_permute_pair_t, METH_FASTCALL,
     "tropical_permute_pair on tensor objects"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_fastcall", "hot entry points of the C ABI", -1,
                                    methods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__fastcall(void)
{
    s_data_ptr = PyUnicode_InternFromString("data_ptr");
    s_shape = PyUnicode_InternFromString("shape");
    s_stride = PyUnicode_InternFromString("stride");
    s_dtype = PyUnicode_InternFromString("dtype");
    s_get_device = PyUnicode_InternFromString("get_device");
    s_cuda_stream = PyUnicode_InternFromString("cuda_stream");
    if (!s_data_ptr || !s_shape || !s_stride || !s_dtype || !s_get_device || !s_cuda_stream) return NULL;
    return PyModule_Create(&module);
}
