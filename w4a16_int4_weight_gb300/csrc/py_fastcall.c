/*
 * Argument marshalling for the Python binding's per-call entry points.
 *
 * ctypes converts each of w4a16_gemm_ex's fourteen arguments through its
 * argtypes on every call, about 1.5 us of host time on a Grace CPU core, close
 * to the CUDA launch itself.  This module takes the same integer
 * arguments with METH_FASTCALL and calls the C ABI function directly.  It does
 * no arithmetic of the layer: addresses and sizes go through unchanged, and the
 * function pointers come from the ctypes-loaded libw4a16 (bind()), so both
 * paths call the same library.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <limits.h>
#include <stdint.h>

typedef int (*gemm_ex_fn)(const void* A, const void* Wq, const void* scales, const int32_t* zeros,
                          const void* Wdense, void* C, int64_t M, int64_t N, int64_t K, int G,
                          int qtype, int dtype, int path, void* stream);
typedef int (*linear_fn)(const void* A, int64_t lda, const void* Wq, const void* scales,
                         const int32_t* zeros, const void* bias, const void* Wdense, void* C,
                         int64_t ldc, int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                         int path, void* stream);

static gemm_ex_fn g_gemm_ex = NULL;
static linear_fn g_linear = NULL;
static PyObject* g_data_ptr = NULL;   /* interned "data_ptr" */

/* None -> NULL; an int -> that address; any other object (a torch tensor) ->
   the address its data_ptr() method returns. */
static void* as_ptr(PyObject* o) {
    if (o == Py_None) return NULL;
    if (PyLong_Check(o)) return PyLong_AsVoidPtr(o);
    if (PyErr_Occurred()) return NULL;   /* an earlier argument failed: call nothing more */
    PyObject* r = PyObject_CallMethodNoArgs(o, g_data_ptr);
    if (!r) return NULL;
    void* p = PyLong_AsVoidPtr(r);
    Py_DECREF(r);
    return p;
}

/* A Python int that fits a C int; OverflowError (set, returns 0) otherwise,
   where a plain cast would keep only the low bits. */
static int as_int(PyObject* o) {
    const long v = PyLong_AsLong(o);
    if (v == -1 && PyErr_Occurred()) return 0;
    if (v < INT_MIN || v > INT_MAX) {
        PyErr_Format(PyExc_OverflowError, "%ld does not fit a 32-bit C integer", v);
        return 0;
    }
    return (int)v;
}

static PyObject* fc_bind(PyObject* self, PyObject* args) {
    unsigned long long gemm_ex = 0, linear = 0;
    (void)self;
    if (!PyArg_ParseTuple(args, "KK", &gemm_ex, &linear)) return NULL;
    if (!gemm_ex || !linear) {
        PyErr_SetString(PyExc_ValueError, "null function address");
        return NULL;
    }
    g_gemm_ex = (gemm_ex_fn)(uintptr_t)gemm_ex;
    g_linear = (linear_fn)(uintptr_t)linear;
    Py_RETURN_NONE;
}

/* gemm_ex(A, Wq, scales, zeros, Wdense, C, M, N, K, G, qtype, dtype, path, stream) -> status */
static PyObject* fc_gemm_ex(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    if (n != 14) {
        PyErr_SetString(PyExc_TypeError, "gemm_ex takes 14 arguments");
        return NULL;
    }
    if (!g_gemm_ex) {
        PyErr_SetString(PyExc_RuntimeError, "bind() was not called");
        return NULL;
    }
    const void* A = as_ptr(a[0]);
    const void* Wq = as_ptr(a[1]);
    const void* scales = as_ptr(a[2]);
    const int32_t* zeros = (const int32_t*)as_ptr(a[3]);
    const void* Wdense = as_ptr(a[4]);
    void* C = as_ptr(a[5]);
    const int64_t M = PyLong_AsLongLong(a[6]), N = PyLong_AsLongLong(a[7]), K = PyLong_AsLongLong(a[8]);
    const int G = as_int(a[9]), qtype = as_int(a[10]), dtype = as_int(a[11]), path = as_int(a[12]);
    void* stream = as_ptr(a[13]);
    if (PyErr_Occurred()) return NULL;
    int st;
    Py_BEGIN_ALLOW_THREADS
    st = g_gemm_ex(A, Wq, scales, zeros, Wdense, C, M, N, K, G, qtype, dtype, path, stream);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(st);
}

/* linear(A, lda, Wq, scales, zeros, bias, Wdense, C, ldc, M, N, K, G, qtype, dtype, path, stream) */
static PyObject* fc_linear(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    if (n != 17) {
        PyErr_SetString(PyExc_TypeError, "linear takes 17 arguments");
        return NULL;
    }
    if (!g_linear) {
        PyErr_SetString(PyExc_RuntimeError, "bind() was not called");
        return NULL;
    }
    const void* A = as_ptr(a[0]);
    const int64_t lda = PyLong_AsLongLong(a[1]);
    const void* Wq = as_ptr(a[2]);
    const void* scales = as_ptr(a[3]);
    const int32_t* zeros = (const int32_t*)as_ptr(a[4]);
    const void* bias = as_ptr(a[5]);
    const void* Wdense = as_ptr(a[6]);
    void* C = as_ptr(a[7]);
    const int64_t ldc = PyLong_AsLongLong(a[8]);
    const int64_t M = PyLong_AsLongLong(a[9]), N = PyLong_AsLongLong(a[10]), K = PyLong_AsLongLong(a[11]);
    const int G = as_int(a[12]), qtype = as_int(a[13]), dtype = as_int(a[14]), path = as_int(a[15]);
    void* stream = as_ptr(a[16]);
    if (PyErr_Occurred()) return NULL;
    int st;
    Py_BEGIN_ALLOW_THREADS
    st = g_linear(A, lda, Wq, scales, zeros, bias, Wdense, C, ldc, M, N, K, G, qtype, dtype, path, stream);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(st);
}

static PyMethodDef fc_methods[] = {
    {"bind", fc_bind, METH_VARARGS, "bind(gemm_ex_address, linear_address)"},
    {"gemm_ex", (PyCFunction)(void (*)(void))fc_gemm_ex, METH_FASTCALL,
     "w4a16_gemm_ex; buffers as None, int addresses or tensors (data_ptr()); returns the status code"},
    {"linear", (PyCFunction)(void (*)(void))fc_linear, METH_FASTCALL,
     "w4a16_linear; buffers as None, int addresses or tensors (data_ptr()); returns the status code"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef fc_module = {PyModuleDef_HEAD_INIT, "_w4a16_fastcall", NULL, -1, fc_methods,
                                       NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__w4a16_fastcall(void) {
    g_data_ptr = PyUnicode_InternFromString("data_ptr");
    if (!g_data_ptr) return NULL;
    return PyModule_Create(&fc_module);
}
