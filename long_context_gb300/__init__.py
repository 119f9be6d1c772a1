"""cpattn: context-parallel ring attention for one GB300 (sm_103a).

Submodules:

* ``long_context_gb300.cpattn``    -- the Python binding of ``libcpattn.so``
  (``plan``, ``fwd``, ``fwd_partials``, ``merge``, ``poll_error``);
* ``long_context_gb300.build``     -- compiles ``libcpattn.so`` with nvcc;
* ``long_context_gb300.workloads`` -- seeded synthetic inputs.

Importing the package itself loads nothing native; importing ``cpattn`` does,
and fails if the library has not been built.
"""
