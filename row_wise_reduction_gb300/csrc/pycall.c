/*
 * _rowops_call: the Python binding's calls into librowops.so for the entry
 * points whose small, launch-bound calls are dominated by host time. It only
 * marshals arguments: Python ints and floats become the C ABI's pointers,
 * sizes and scalars, the call runs with the GIL released, and its status comes
 * back as an int. The function addresses are handed over once by the ctypes
 * loader (bind), so this module does not link the library itself.
 *
 * A ctypes call with seven typed arguments costs about 2 us of Python time;
 * through this module, about 0.1 us.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stdint.h>

typedef int (*softmax_fn)(const void*, void*, int64_t, int64_t, int64_t, int, void*);
typedef int (*ln_fn)(const void*, void*, const void*, const void*, float, int64_t, int64_t, int64_t, int, void*);

static softmax_fn g_softmax = NULL;
static ln_fn g_ln = NULL;
static ln_fn g_ln_erf = NULL;

static int as_ptr(PyObject* o, void** out) {
    if (o == Py_None) {
        *out = NULL;
        return 0;
    }
    *out = PyLong_AsVoidPtr(o);
    return (*out == NULL && PyErr_Occurred()) ? -1 : 0;
}

static int as_i64(PyObject* o, int64_t* out) {
    long long v = PyLong_AsLongLong(o);
    if (v == -1 && PyErr_Occurred()) return -1;
    *out = (int64_t)v;
    return 0;
}

static int nargs_ok(Py_ssize_t n, Py_ssize_t want, const char* name) {
    if (n == want) return 1;
    PyErr_Format(PyExc_TypeError, "%s takes %zd arguments (%zd given)", name, want, n);
    return 0;
}

/* bind(softmax, layernorm_gelu, layernorm_gelu_erf): function addresses */
static PyObject* bind(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    void *s, *l, *e;
    (void)self;
    if (!nargs_ok(n, 3, "bind") || as_ptr(a[0], &s) || as_ptr(a[1], &l) || as_ptr(a[2], &e)) return NULL;
    g_softmax = (softmax_fn)s;
    g_ln = (ln_fn)l;
    g_ln_erf = (ln_fn)e;
    Py_RETURN_NONE;
}

/* softmax(x, y, M, N, ld, dtype, stream) -> status */
static PyObject* softmax(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    void *x, *y, *st;
    int64_t M, N, ld, dt;
    int r;
    (void)self;
    if (!g_softmax) return PyErr_Format(PyExc_RuntimeError, "_rowops_call is not bound");
    if (!nargs_ok(n, 7, "softmax") || as_ptr(a[0], &x) || as_ptr(a[1], &y) || as_i64(a[2], &M) ||
        as_i64(a[3], &N) || as_i64(a[4], &ld) || as_i64(a[5], &dt) || as_ptr(a[6], &st))
        return NULL;
    Py_BEGIN_ALLOW_THREADS
    r = g_softmax(x, y, M, N, ld, (int)dt, st);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(r);
}

static PyObject* ln_call(ln_fn f, const char* name, PyObject* const* a, Py_ssize_t n) {
    void *x, *y, *w, *b, *st;
    int64_t M, N, ld, dt;
    double eps;
    int r;
    if (!f) return PyErr_Format(PyExc_RuntimeError, "_rowops_call is not bound");
    if (!nargs_ok(n, 10, name) || as_ptr(a[0], &x) || as_ptr(a[1], &y) || as_ptr(a[2], &w) || as_ptr(a[3], &b))
        return NULL;
    eps = PyFloat_AsDouble(a[4]);
    if (eps == -1.0 && PyErr_Occurred()) return NULL;
    if (as_i64(a[5], &M) || as_i64(a[6], &N) || as_i64(a[7], &ld) || as_i64(a[8], &dt) || as_ptr(a[9], &st))
        return NULL;
    Py_BEGIN_ALLOW_THREADS
    r = f(x, y, w, b, (float)eps, M, N, ld, (int)dt, st);
    Py_END_ALLOW_THREADS
    return PyLong_FromLong(r);
}

/* layernorm_gelu(x, y, w, b, eps, M, N, ld, dtype, stream) -> status (w, b may be None) */
static PyObject* layernorm_gelu(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    return ln_call(g_ln, "layernorm_gelu", a, n);
}

static PyObject* layernorm_gelu_erf(PyObject* self, PyObject* const* a, Py_ssize_t n) {
    (void)self;
    return ln_call(g_ln_erf, "layernorm_gelu_erf", a, n);
}

static PyMethodDef methods[] = {
    {"bind", (PyCFunction)(void (*)(void))bind, METH_FASTCALL, "bind(softmax, layernorm_gelu, layernorm_gelu_erf)"},
    {"softmax", (PyCFunction)(void (*)(void))softmax, METH_FASTCALL, "rowops_softmax"},
    {"layernorm_gelu", (PyCFunction)(void (*)(void))layernorm_gelu, METH_FASTCALL, "rowops_layernorm_gelu"},
    {"layernorm_gelu_erf", (PyCFunction)(void (*)(void))layernorm_gelu_erf, METH_FASTCALL,
     "rowops_layernorm_gelu_erf"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_rowops_call", NULL, -1, methods,
                                    NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__rowops_call(void) { return PyModule_Create(&module); }
