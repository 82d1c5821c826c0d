/* gemm_pycall.c -- CPython entry points for the two per-call functions of the
 * C ABI, gemm_run and gemm_launch_empty: one vectorcall with plain integer
 * arguments instead of a ctypes call that converts each argument.  Argument
 * marshalling only: the functions are called through the addresses the Python
 * binding hands over once, after it has loaded libgemm_gb300.so.
 *
 *   set_targets(run_address, empty_address)
 *   run(plan, a, b, c, stream) -> gemm_status_t   (addresses as Python ints)
 *   launch_empty(grid, stream) -> gemm_status_t
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>

typedef int (*gemm_run_fn)(void*, const void*, const void*, void*, void*);
typedef int (*gemm_launch_empty_fn)(int, void*);

static gemm_run_fn g_run = NULL;
static gemm_launch_empty_fn g_empty = NULL;

static PyObject* set_targets(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 2) {
        PyErr_SetString(PyExc_TypeError, "set_targets(run_address, empty_address)");
        return NULL;
    }
    void* run = PyLong_AsVoidPtr(args[0]);
    if (run == NULL && PyErr_Occurred()) return NULL;
    void* empty = PyLong_AsVoidPtr(args[1]);
    if (empty == NULL && PyErr_Occurred()) return NULL;
    g_run = (gemm_run_fn)run;
    g_empty = (gemm_launch_empty_fn)empty;
    Py_RETURN_NONE;
}

static PyObject* run(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 5) {
        PyErr_SetString(PyExc_TypeError, "run(plan, a, b, c, stream)");
        return NULL;
    }
    if (g_run == NULL) {
        PyErr_SetString(PyExc_RuntimeError, "gemm_run address not set");
        return NULL;
    }
    void* v[5];
    for (int i = 0; i < 5; ++i) {
        v[i] = PyLong_AsVoidPtr(args[i]);   /* 0 -> NULL without an error */
        if (v[i] == NULL && PyErr_Occurred()) return NULL;
    }
    return PyLong_FromLong(g_run(v[0], v[1], v[2], v[3], v[4]));
}

static PyObject* launch_empty(PyObject* self, PyObject* const* args, Py_ssize_t nargs) {
    (void)self;
    if (nargs != 2) {
        PyErr_SetString(PyExc_TypeError, "launch_empty(grid, stream)");
        return NULL;
    }
    if (g_empty == NULL) {
        PyErr_SetString(PyExc_RuntimeError, "gemm_launch_empty address not set");
        return NULL;
    }
    const long grid = PyLong_AsLong(args[0]);
    if (grid == -1 && PyErr_Occurred()) return NULL;
    void* stream = PyLong_AsVoidPtr(args[1]);
    if (stream == NULL && PyErr_Occurred()) return NULL;
    return PyLong_FromLong(g_empty((int)grid, stream));
}

static PyMethodDef methods[] = {
    {"set_targets", (PyCFunction)(void (*)(void))set_targets, METH_FASTCALL,
     "set_targets(run_address, empty_address)"},
    {"run", (PyCFunction)(void (*)(void))run, METH_FASTCALL,
     "run(plan, a, b, c, stream) -> status of gemm_run"},
    {"launch_empty", (PyCFunction)(void (*)(void))launch_empty, METH_FASTCALL,
     "launch_empty(grid, stream) -> status of gemm_launch_empty"},
    {NULL, NULL, 0, NULL},
};

static struct PyModuleDef module = {PyModuleDef_HEAD_INIT, "_gemm_pycall",
                                    "Vectorcall entry points for gemm_run and gemm_launch_empty.",
                                    -1, methods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__gemm_pycall(void) { return PyModule_Create(&module); }
