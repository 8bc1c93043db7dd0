"""The oracle: a plain, slow, obviously correct CPU statement of the decoder step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this package:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may use it. It shares no code, header, table or constant generator with the
CUDA library; the two meet only through the seeded inputs of the ``synth`` package.

Every floating-point definition is evaluated in float64 from float32 inputs, with numpy
and a BLAS matrix product as the only library primitives, and no blocking, fusion or
reordering beyond what each definition states. The one exception is the embedding
backward, whose scatter-add is defined in float32 in ascending row order so that an exact
(bit-identical) comparison has a meaning.

Sources, cited in each docstring by these short tags (page title, then section):

[LM1] arabroot.io, "Build a language model in C# from scratch (1): the Autograd engine".
[LM4] arabroot.io, "Build a language model in C# from scratch (4): running GPT-2 weights".
[AD]  nextadmin.net, "Chain rule and automatic differentiation: implementing Autograd
      from scratch".

Readings taken where the pages are silent are stated at the function they affect.
"""
