/* gemm_pycall.c -- CPython entry points for the two per-call functions of the
 * C ABI, gemm_run and gemm_launch_empty: one vectorcall with plain integer
 * arguments instead of a ctypes call that converts each argument.  Argument
 * marshalling only: the functions are called through the addresses the Python
 * binding hands over once, after it has loaded libgemm_gb300.so.
 *
 *   set_targets(run_address, empty_address)
 *   run(plan, a, b, c, stream) -> gemm_status_t   (addresses as Python ints)
 *   launch_empty(grid, stream) -> gemm_status_t
 *   Runner(box, general) -> a callable for one plan: runner(A, B, C, stream)
 *       with three objects that have a data_ptr() method (torch tensors) and a
 *       stream object with a cuda_stream attribute calls gemm_run(box[0], ...)
 *       directly; every other call, a box[0] that is None (plan closed) and a
 *       non-zero status go to general(*args, **kwargs), the binding's own path,
 *       which handles the other argument forms and raises the error.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <stddef.h>

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

typedef struct {
    PyObject_HEAD
    PyObject* box;       /* list whose item 0 is the plan handle (an int) or None */
    PyObject* general;   /* fallback callable */
    vectorcallfunc vectorcall;
} Runner;

static PyObject* s_data_ptr = NULL;
static PyObject* s_cuda_stream = NULL;

/* The address an object reports, or NULL (error cleared) if it has none. */
static int address_of(PyObject* obj, PyObject* name, int is_method, void** out) {
    PyObject* r = is_method ? PyObject_VectorcallMethod(name, &obj, 1, NULL)
                            : PyObject_GetAttr(obj, name);
    if (r == NULL) {
        PyErr_Clear();
        return 0;
    }
    *out = PyLong_AsVoidPtr(r);
    Py_DECREF(r);
    if (*out == NULL && PyErr_Occurred()) {
        PyErr_Clear();
        return 0;
    }
    return 1;
}

static PyObject* runner_call(PyObject* self_, PyObject* const* args, size_t nargsf,
                             PyObject* kwnames) {
    Runner* self = (Runner*)self_;
    const Py_ssize_t nargs = PyVectorcall_NARGS(nargsf);
    if (nargs == 4 && kwnames == NULL && g_run != NULL) {
        PyObject* h = PyList_GET_ITEM(self->box, 0);
        void* plan = h == Py_None ? NULL : PyLong_AsVoidPtr(h);
        if (plan == NULL) PyErr_Clear();
        void* v[4];
        if (plan != NULL && address_of(args[0], s_data_ptr, 1, &v[0]) &&
            address_of(args[1], s_data_ptr, 1, &v[1]) &&
            address_of(args[2], s_data_ptr, 1, &v[2]) &&
            address_of(args[3], s_cuda_stream, 0, &v[3]) &&
            g_run(plan, v[0], v[1], v[2], v[3]) == 0)
            Py_RETURN_NONE;
    }
    return PyObject_Vectorcall(self->general, args, nargsf, kwnames);
}

static PyObject* runner_new(PyTypeObject* type, PyObject* args, PyObject* kwds) {
    PyObject *box, *general;
    if (kwds != NULL && PyDict_GET_SIZE(kwds) != 0) {
        PyErr_SetString(PyExc_TypeError, "Runner(box, general)");
        return NULL;
    }
    if (!PyArg_ParseTuple(args, "O!O:Runner", &PyList_Type, &box, &general)) return NULL;
    if (PyList_GET_SIZE(box) < 1 || !PyCallable_Check(general)) {
        PyErr_SetString(PyExc_TypeError, "Runner(box, general): a non-empty list and a callable");
        return NULL;
    }
    Runner* self = (Runner*)type->tp_alloc(type, 0);
    if (self == NULL) return NULL;
    Py_INCREF(box);
    Py_INCREF(general);
    self->box = box;
    self->general = general;
    self->vectorcall = runner_call;
    return (PyObject*)self;
}

static int runner_traverse(PyObject* self_, visitproc visit, void* arg) {
    Runner* self = (Runner*)self_;
    Py_VISIT(self->box);
    Py_VISIT(self->general);
    return 0;
}

static int runner_clear(PyObject* self_) {
    Runner* self = (Runner*)self_;
    Py_CLEAR(self->box);
    Py_CLEAR(self->general);
    return 0;
}

static void runner_dealloc(PyObject* self) {
    PyObject_GC_UnTrack(self);
    runner_clear(self);
    Py_TYPE(self)->tp_free(self);
}

static PyTypeObject RunnerType = {
    PyVarObject_HEAD_INIT(NULL, 0)
    .tp_name = "_gemm_pycall.Runner",
    .tp_basicsize = sizeof(Runner),
    .tp_flags = Py_TPFLAGS_DEFAULT | Py_TPFLAGS_HAVE_GC | Py_TPFLAGS_HAVE_VECTORCALL,
    .tp_doc = "Runner(box, general): gemm_run for one plan, called as runner(A, B, C, stream)",
    .tp_new = runner_new,
    .tp_dealloc = runner_dealloc,
    .tp_traverse = runner_traverse,
    .tp_clear = runner_clear,
    .tp_call = PyVectorcall_Call,
    .tp_vectorcall_offset = offsetof(Runner, vectorcall),
};

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
                                    "Vectorcall entry points for gemm_run and gemm_launch_empty, "
                                    "and a per-plan runner.",
                                    -1, methods, NULL, NULL, NULL, NULL};

PyMODINIT_FUNC PyInit__gemm_pycall(void) {
    s_data_ptr = PyUnicode_InternFromString("data_ptr");
    s_cuda_stream = PyUnicode_InternFromString("cuda_stream");
    if (s_data_ptr == NULL || s_cuda_stream == NULL || PyType_Ready(&RunnerType) < 0) return NULL;
    PyObject* m = PyModule_Create(&module);
    if (m == NULL) return NULL;
    Py_INCREF(&RunnerType);
    if (PyModule_AddObject(m, "Runner", (PyObject*)&RunnerType) < 0) {
        Py_DECREF(&RunnerType);
        Py_DECREF(m);
        return NULL;
    }
    return m;
}
