"""GB300-native (sm_103a) DDTree verify step: best-first draft-tree build,
tree-verify MLA-absorb attention, greedy accept and cache compaction, exposed
through the C ABI in ``include/ddt.h`` and the thin ctypes binding in
:mod:`._binding`."""
